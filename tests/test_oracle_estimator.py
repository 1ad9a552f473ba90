"""Pins for the asymmetric estimator: unbiasedness, variance, limits."""
from math import pi, sqrt

import numpy as np

import oracle
from oracle import rng
from oracle.codebook import sphere_codebook


def _fixed_xq(d):
    x = rng.gaussian_stream(1001, d)
    q = rng.gaussian_stream(1002, d)
    return x, q


def test_unbiased_over_seeds():
    # "Zero-bias" (freelamp article, QJL section) / "unbiased estimate" (csdn tutorial, QJL
    # step 3): over fresh (Pi, S) draws the mean of est - <q, x> is 0 within 3 SE.
    d, n = 16, 6000
    x, q = _fixed_xq(d)
    cb = sphere_codebook(d, 1)
    err = np.empty(n)
    for s in range(n):
        Pi, S = rng.method_matrices(10_000 + s, d, d)
        z = oracle.quantize(x[None], Pi, cb, S)
        err[s] = oracle.estimate(q, z, Pi, cb, S)[0] - q @ x
    se = err.std() / np.sqrt(n)
    assert abs(err.mean()) < 3 * se
    # the MSE-only estimate is biased (shrunk towards 0): the correction matters
    mse_only = np.empty(400)
    for s in range(400):
        Pi, _ = rng.method_matrices(20_000 + s, d, 1)
        z = oracle.quantize(x[None], Pi, cb)
        mse_only[s] = oracle.estimate(q, z, Pi, cb)[0] - q @ x
    assert abs(mse_only.mean()) > 5 * mse_only.std() / np.sqrt(400)


def test_qjl_term_conditional_mean_and_variance():
    # Pi fixed, S fresh: the correction has mean <q, r> and variance
    # (pi/2 ||r||^2 ||q||^2 - <q, r>^2) / m.  A wrong constant (sqrt(2/pi) for sqrt(pi/2))
    # or a flipped sign convention moves the mean by many SE.
    d, m, n = 16, 16, 20000
    x, _ = _fixed_xq(d)
    Pi, _ = rng.method_matrices(5, d, 1)
    cb = sphere_codebook(d, 1)
    z0 = oracle.quantize(x[None], Pi, cb)
    r = x - oracle.dequantize(z0.idx, z0.norm16, Pi, cb)[0]
    q = r + 0.3 * rng.gaussian_stream(77, d)
    rn = np.linalg.norm(r)
    terms = np.empty(n)
    for s in range(n):
        S = rng.jl_matrix(40_000 + s, m, d)
        signs = (S @ r) > 0
        terms[s] = rn * sqrt(pi / 2) / m * ((2.0 * signs - 1.0) @ (S @ q))
    se = terms.std() / np.sqrt(n)
    assert abs(terms.mean() - q @ r) < 3 * se
    var = (pi / 2 * rn ** 2 * (q @ q) - (q @ r) ** 2) / m
    assert abs(terms.var() / var - 1.0) < 0.05


def test_oracle_estimate_uses_stored_rnorm():
    # The estimator's correction equals the conditional-mean construction above when
    # rnorm16 is the residual norm; check est = <q, x_hat> + correction term by term.
    d = 32
    Pi, S = rng.method_matrices(6, d, d)
    cb = sphere_codebook(d, 2)
    X = rng.gaussian_stream(7, 10 * d).reshape(10, d)
    q = rng.gaussian_stream(8, d)
    z = oracle.quantize(X, Pi, cb, S)
    xhat = oracle.dequantize(z.idx, z.norm16, Pi, cb)
    corr = z.rnorm16 * sqrt(pi / 2) / d * ((2.0 * z.signs - 1.0) @ (S @ q))
    assert np.allclose(oracle.estimate(q, z, Pi, cb, S), xhat @ q + corr, rtol=1e-12, atol=1e-12)


def test_large_m_correction_tends_to_residual_product():
    d, m = 16, 200000
    x, q = _fixed_xq(d)
    Pi, _ = rng.method_matrices(9, d, 1)
    S = rng.jl_matrix(123, m, d)
    cb = sphere_codebook(d, 2)
    z = oracle.quantize(x[None], Pi, cb, S)
    r = x - oracle.dequantize(z.idx, z.norm16, Pi, cb)[0]
    est = oracle.estimate(q, z, Pi, cb, S)[0]
    xhat_q = oracle.dequantize(z.idx, z.norm16, Pi, cb)[0] @ q
    sd = sqrt((pi / 2 * (r @ r) * (q @ q)) / m)
    # rnorm16 carries a relative fp16 rounding of at most 2^-11
    assert abs((est - xhat_q) - q @ r) < 4 * sd + 2 ** -11 * abs(q @ r)


def test_inner_product_distortion_falls_with_bits():
    d, n = 32, 3000
    Pi, S = rng.method_matrices(12, d, d)
    X = rng.gaussian_stream(13, n * d).reshape(n, d)
    q = rng.gaussian_stream(14, d)
    prev = np.inf
    for bits in (1, 2, 3):
        cb = sphere_codebook(d, bits)
        z = oracle.quantize(X, Pi, cb, S)
        e = np.mean((oracle.estimate(q, z, Pi, cb, S) - X @ q) ** 2)
        assert e < prev
        prev = e
