"""Pins for the fractional-bit-width oracle (juejin.cn post section 四: KV quality stated at 3.5
and 2.5 bits per channel).  The reading: the first d_hi rotated coordinates use the (b+1)-bit
Lloyd-Max table, the rest the b-bit table.  Each pin checks the split code against something
other than itself: the uniform tables it must reduce to, brute-force nearest centroids, the
closed-form distortion of each table, unbiasedness over seeds, and the packed layout bit by
bit."""
import numpy as np
import pytest

import oracle
from oracle import rng
from oracle.codebook import sphere_codebook


def _split(d, b, d_hi):
    return oracle.SplitCodebook(lo=sphere_codebook(d, b), hi=sphere_codebook(d, b + 1), d_hi=d_hi)


@pytest.mark.parametrize("b", [1, 2, 3])
def test_split_reduces_to_the_uniform_tables(b):
    d = 64
    Pi, S = rng.method_matrices(7, d, d)
    X = rng.gaussian_stream(8, 300 * d).reshape(300, d)
    for d_hi, cb in ((0, sphere_codebook(d, b)), (d, sphere_codebook(d, b + 1))):
        scb = _split(d, b, d_hi)
        zs, zu = oracle.split_quantize(X, Pi, scb, S), oracle.quantize(X, Pi, cb, S)
        assert np.array_equal(zs.idx, zu.idx)
        assert np.array_equal(zs.signs, zu.signs)
        assert np.array_equal(zs.rnorm16, zu.rnorm16) and np.array_equal(zs.norm16, zu.norm16)
        q = rng.gaussian_stream(9, d)
        assert np.allclose(oracle.split_estimate(q, zs, Pi, scb, S), oracle.estimate(q, zu, Pi, cb, S), rtol=0, atol=1e-12)


def test_split_codes_are_the_nearest_centroid_of_each_coordinate_table():
    d, b, d_hi = 32, 2, 8
    scb = _split(d, b, d_hi)
    U = rng.gaussian_stream(10, 500 * d).reshape(500, d) * 0.3
    idx = scb.codes(U)
    for j in range(d):
        c = (scb.hi if j < d_hi else scb.lo).centroids
        brute = np.argmin(np.abs(U[:, j, None] - c[None, :]), axis=1)
        assert np.array_equal(idx[:, j], brute)
    assert idx[:, :d_hi].max() <= 2 ** (b + 1) - 1 and idx[:, d_hi:].max() <= 2 ** b - 1


@pytest.mark.parametrize("b,d_hi", [(1, 32), (2, 32), (2, 16)])
def test_split_distortion_is_the_coordinate_average_of_the_two_tables(b, d_hi):
    # E ||u - c_g[idx]||^2 = (d_hi / d) D(b+1) + (1 - d_hi / d) D(b), D the closed-form
    # distortion of each table (pinned in test_oracle_codebook.py); Monte Carlo within 3 SE.
    d, n = 64, 4000
    scb = _split(d, b, d_hi)
    Pi, _ = rng.method_matrices(11, d, 1)
    X = rng.gaussian_stream(12, n * d).reshape(n, d)
    U = (X @ Pi.T) / np.linalg.norm(X, axis=1, keepdims=True)
    err = ((U - scb.centroid_values(scb.codes(U))) ** 2).sum(axis=1)
    want = (d_hi / d) * scb.hi.distortion() + (1 - d_hi / d) * scb.lo.distortion()
    assert abs(err.mean() - want) < 3 * err.std() / np.sqrt(n)
    # and it lies strictly between the two uniform widths
    assert scb.hi.distortion() < err.mean() < scb.lo.distortion()


def test_split_estimator_is_unbiased_over_seeds():
    d, n, b, d_hi = 16, 5000, 1, 8
    scb = _split(d, b, d_hi)
    x, q = rng.gaussian_stream(1001, d), rng.gaussian_stream(1002, d)
    err = np.empty(n)
    for s in range(n):
        Pi, S = rng.method_matrices(30_000 + s, d, d)
        z = oracle.split_quantize(x[None], Pi, scb, S)
        err[s] = oracle.split_estimate(q, z, Pi, scb, S)[0] - q @ x
    assert abs(err.mean()) < 3 * err.std() / np.sqrt(n)


@pytest.mark.parametrize("d,b,d_hi", [(128, 2, 64), (128, 1, 32), (100, 3, 64)])
def test_split_packing_layout(d, b, d_hi):
    g = np.random.default_rng(5)
    idx = np.concatenate([g.integers(0, 2 ** (b + 1), size=(7, d_hi)), g.integers(0, 2 ** b, size=(7, d - d_hi))], axis=1)
    words = oracle.pack_split(idx, b, d_hi)
    W, Wh = (d + 31) // 32, (d_hi + 31) // 32
    assert words.shape == (7, b * W + Wh) and words.dtype == np.uint32
    assert np.array_equal(oracle.unpack_split(words, d, b, d_hi), idx)
    for r, j in [(0, 0), (3, d_hi - 1), (6, d - 1), (2, 31)]:
        for p in range(b):
            assert (int(words[r, p * W + j // 32]) >> (j % 32)) & 1 == (idx[r, j] >> p) & 1
        if j < d_hi:
            assert (int(words[r, b * W + j // 32]) >> (j % 32)) & 1 == (idx[r, j] >> b) & 1
