"""Pins for the oracle's PolarQuant stage, residual, QJL signs and packing."""
import numpy as np
import pytest

import oracle
from oracle import rng
from oracle.codebook import sphere_codebook
from oracle.turboquant import scalar_codes
from conftest import read_golden


def _unit_rows(n, d, seed):
    g = rng.gaussian_stream(seed, n * d).reshape(n, d)
    return g / np.linalg.norm(g, axis=1, keepdims=True)


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 6, 8])
def test_threshold_count_is_brute_force_nearest(bits):
    cb = sphere_codebook(12, bits)
    u = rng.gaussian_stream(5, 5000) / np.sqrt(12)
    nearest = np.argmin(np.abs(u[:, None] - cb.centroids[None, :]), axis=1)
    assert np.array_equal(scalar_codes(u, cb), nearest)


def test_value_on_threshold_takes_lower_index():
    cb = sphere_codebook(32, 3)
    assert np.array_equal(scalar_codes(cb.thresholds, cb), np.arange(len(cb.thresholds)))


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
def test_centroids_round_trip(bits):
    # Each centroid lies inside its own cell: coding a codebook value returns its index,
    # so dequantize-then-code is the identity on the codes.
    cb = sphere_codebook(64, bits)
    assert np.array_equal(scalar_codes(cb.centroids, cb), np.arange(cb.levels))


def test_mse_matches_table_and_falls_with_bits():
    # "MSE falls as the bit width grows" (juejin.cn post, section 四): the empirical
    # E||u - c[idx]||^2 over random unit vectors equals the table's D(b) within 3 SE.
    d, n = 16, 100000
    Pi, _ = rng.method_matrices(1, d, 1)
    X = rng.gaussian_stream(2, n * d).reshape(n, d)
    emp = []
    for bits in range(1, 9):
        cb = sphere_codebook(d, bits)
        z = oracle.quantize(X, Pi, cb)
        U = (X @ Pi.T) / np.linalg.norm(X, axis=1, keepdims=True)
        err = np.sum((U - cb.centroids[z.idx]) ** 2, axis=1)
        assert abs(err.mean() - cb.distortion()) < 3 * err.std() / np.sqrt(n)
        emp.append(err.mean())
    assert all(emp[i + 1] < emp[i] for i in range(7))


@pytest.mark.parametrize("d", [128, 200])
def test_round_trip_at_eight_bits(d):
    # "Exact round trip at high bit width" (juejin.cn post, section 四), read at b_m = 8 MSE bits.
    # Coding the reconstruction x_hat = n16 Pi^T c[idx] again sees the direction c[idx] / |c[idx]|,
    # every centroid scaled by 1 / |c[idx]|.  Where |c[idx]| = 1 to within 5e-3 (over 99 % of rows)
    # that keeps each centroid inside its cell, so the codes come back unchanged; a row with a
    # coordinate far beyond the outermost centroid has |c[idx]| further from 1 and may re-code
    # differently (the renormalisation moves values across thresholds).  The relative reconstruction
    # error is the
    # table's distortion: mean |x - x_hat|^2 / |x|^2 = D(8) within 3 SE (plus the fp16 norm's at
    # most 2^-22 relative square error).
    n = 4000
    Pi, _ = rng.method_matrices(3, d, 1)
    cb = sphere_codebook(d, 8)
    X = 5.0 * rng.gaussian_stream(11, n * d).reshape(n, d)
    z = oracle.quantize(X, Pi, cb)
    Xh = oracle.dequantize(z.idx, z.norm16, Pi, cb)
    z2 = oracle.quantize(Xh, Pi, cb)
    unit = np.abs(np.linalg.norm(cb.centroids[z.idx], axis=1) - 1.0) < 5e-3
    assert unit.mean() > 0.99
    assert np.array_equal(z2.idx[unit], z.idx[unit])
    rel = np.sum((X - Xh) ** 2, axis=1) / np.sum(X ** 2, axis=1)
    assert abs(rel.mean() - cb.distortion()) < 3 * rel.std() / np.sqrt(n) + 2.0 ** -22
    assert np.median(np.sqrt(rel)) < 1.2 * np.sqrt(cb.distortion())


def test_reconstruction_error_and_norm():
    d, n = 64, 4000
    Pi, _ = rng.method_matrices(4, d, 1)
    X = 3.0 * rng.gaussian_stream(5, n * d).reshape(n, d)
    cb = sphere_codebook(d, 4)
    z = oracle.quantize(X, Pi, cb)
    assert np.array_equal(z.norm16, np.linalg.norm(X, axis=1).astype(np.float16).astype(np.float64))
    rel = np.sum((X - oracle.dequantize(z.idx, z.norm16, Pi, cb)) ** 2, axis=1) / np.sum(X ** 2, axis=1)
    # fp16 norm adds at most ~2^-11 relative error on top of the codebook distortion
    assert abs(rel.mean() - cb.distortion()) < 3 * rel.std() / np.sqrt(n) + 1e-5


def test_zero_vector():
    d = 8
    Pi, S = rng.method_matrices(0, d, d)
    cb = sphere_codebook(d, 2)
    z = oracle.quantize(np.zeros((1, d)), Pi, cb, S)
    assert z.norm16[0] == 0 and z.rnorm16[0] == 0 and not z.signs.any()
    assert np.all(z.idx == len(cb.thresholds) // 2)   # u = 0 sits on the middle threshold -> lower index


def test_sign_convention_and_residual():
    g = read_golden("bit_budget.txt")
    d = 16
    Pi, _ = rng.method_matrices(8, d, 1)
    cb = sphere_codebook(d, 2)
    X = rng.gaussian_stream(9, 50 * d).reshape(50, d)
    S = np.eye(d)                                       # S = I: sign bits are the residual's signs
    z = oracle.quantize(X, Pi, cb, S)
    R = X - z.norm16[:, None] * (cb.centroids[z.idx] @ Pi)
    assert np.array_equal(z.signs, np.where(R > 0, g["sign_positive_bit"][0], g["sign_negative_bit"][0]).astype(bool))
    assert np.array_equal(z.rnorm16, np.linalg.norm(R, axis=1).astype(np.float16).astype(np.float64))


def test_packing_worked_example():
    g = read_golden("packing_example.txt")
    d = g["d"][0]
    idx = np.arange(d) % 4
    planes = oracle.pack_planes(idx[None, :], 2)[0]
    assert [int(w) for w in planes[0]] == g["plane0"]
    assert [int(w) for w in planes[1]] == g["plane1"]
    assert np.array_equal(oracle.unpack_planes(planes[None], d)[0], idx)


def test_pack_round_trip_random():
    r = np.random.default_rng(0)
    for d in (1, 31, 32, 33, 200):
        idx = r.integers(0, 8, size=(5, d))
        planes = oracle.pack_planes(idx, 3)
        assert planes.shape == (5, 3, (d + 31) // 32)
        assert np.array_equal(oracle.unpack_planes(planes, d), idx)
        s = r.integers(0, 2, size=(5, d)).astype(bool)
        w = oracle.pack_signs(s)
        assert np.array_equal(oracle.unpack_signs(w, d), s)
        if d % 32:
            assert np.all(w[:, -1] >> np.uint32(d % 32) == 0)   # pad bits are 0


def test_bit_budget():
    g = read_golden("bit_budget.txt")
    for mse_bits, total in zip(g["mse_bits"], g["total_bits"]):
        d = 128
        cb = sphere_codebook(d, mse_bits)
        code_bits = d * int(np.log2(cb.levels))
        sign_bits = d                                   # m = d, one bit each
        assert (code_bits + sign_bits) / d == total
    assert np.finfo(np.float16).bits == g["norm_bits"][0]
