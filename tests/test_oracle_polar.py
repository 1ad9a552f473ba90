"""Pins for the recursive polar-angle oracle (csdn tutorial, sections "PolarQuant" and
"将笛卡尔积坐标转为极坐标"; freelamp article, section "技术突破：极坐标量化").  Each pin checks the
oracle against something other than itself: the pages' worked examples, closed forms of the angle
laws and tables, Monte Carlo draws from the laws by another route, brute-force nearest centroids,
unbiasedness over seeds and the packed layout bit by bit."""
from math import pi

import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import rng
from conftest import read_golden


def test_page_2d_example():
    g = read_golden("polar_2d_example.txt")
    r, angles, _ = oracle.polar_forward(np.array([g["legs"]]))
    assert r[0] == pytest.approx(g["r"][0], abs=1e-12)
    assert round(float(np.degrees(angles[0][0, 0]))) == g["angle_deg_rounded"][0]


def test_page_4d_example():
    # the rotated example vector [5, 5, 5, 5]: its radius is |X| = 10 and every angle of equal
    # children is pi / 4
    g = read_golden("p5_rotation_example.txt")
    r, angles, radii = oracle.polar_forward(np.array([g["QX"]]))
    assert r[0] == pytest.approx(np.linalg.norm(g["X"]), abs=1e-12)
    assert len(angles) == 2 and angles[0].shape == (1, 2) and angles[1].shape == (1, 1)
    for a in angles:
        assert np.allclose(a, pi / 4, atol=1e-15)
    assert np.allclose(radii[0], 5 * np.sqrt(2), atol=1e-13)


def test_axis_vectors_and_zero():
    # closed forms: e_0 -> all angles 0; e_1 -> level-1 angle pi/2 in its pair, level-2 angles 0;
    # -e_0 -> level-1 angle pi; the zero vector -> radius 0, every code 0, reconstruction 0
    d = 8
    E = np.zeros((4, d))
    E[0, 0], E[1, 1], E[2, 0], E[3, 5] = 1.0, 1.0, -1.0, 2.0
    r, a, _ = oracle.polar_forward(E)
    assert np.allclose(r, [1, 1, 1, 2])
    assert np.allclose(a[0][0], 0) and np.allclose(a[1][0], 0) and np.allclose(a[2][0], 0)
    assert a[0][1, 0] == pytest.approx(pi / 2) and np.allclose(a[0][1, 1:], 0)
    assert a[0][2, 0] == pytest.approx(pi)
    # coordinate 5 = pair 2 (right child), that pair is the left child of level-2 node 1,
    # which is the right child of the root
    assert a[0][3, 2] == pytest.approx(pi / 2) and a[1][3, 1] == pytest.approx(0.0) and a[2][3, 0] == pytest.approx(pi / 2)
    pcb = oracle.polar_codebook(d, 2)
    Pi = np.eye(d)
    z = oracle.polar_quantize(np.zeros((1, d)), Pi, pcb)
    assert z.r16[0] == 0 and not z.codes.any()
    assert not oracle.polar_dequantize(z.codes, z.r16, Pi, pcb).any()


@pytest.mark.parametrize("d", [2, 4, 16, 128])
def test_inverse_rebuilds_the_vector(d):
    Y = rng.gaussian_stream(40 + d, 200 * d).reshape(200, d)
    r, angles, _ = oracle.polar_forward(Y)
    assert len(angles) == int(np.log2(d)) and sum(a.shape[1] for a in angles) == d - 1
    assert np.allclose(r, np.linalg.norm(Y, axis=1), rtol=1e-14)
    assert np.max(np.abs(oracle.polar_inverse(r, angles) - Y)) < 1e-13


@pytest.mark.parametrize("level", [1, 2, 3, 4, 5])
def test_angle_laws_fit_rotated_gaussian_rows(level):
    # the analytic law of each level against the angles of Gaussian rows (KS at n = 20000)
    d, n = 32, 20000
    Y = rng.gaussian_stream(77, n * d).reshape(n, d)
    _, angles, _ = oracle.polar_forward(Y)
    sample = angles[level - 1][:, 0]
    ks = stats.kstest(sample, lambda t: oracle.angle_cdf(t, level)).statistic
    assert ks < 0.012


def test_density_integrates_to_the_cdf():
    for level in (2, 3, 6):
        t = np.linspace(0, pi / 2, 20001)
        f = oracle.angle_pdf(t, level)
        cum = np.concatenate([[0.0], np.cumsum((f[1:] + f[:-1]) / 2 * np.diff(t))])
        assert np.max(np.abs(cum - oracle.angle_cdf(t, level))) < 1e-7


def test_closed_form_tables():
    # level 2 (k = 2, density sin 2 psi): the 1-bit table splits at pi/4 and its centroids are
    # int_0^{pi/4} psi sin 2psi / int_0^{pi/4} sin 2psi = (1/4) / (1/2) = 1/2 and pi/2 - 1/2
    cb = oracle.angle_codebook(2, 1)
    assert cb.thresholds[0] == pytest.approx(pi / 4, abs=1e-13)
    assert np.allclose(cb.centroids, [0.5, pi / 2 - 0.5], atol=1e-12)
    # level 1: the uniform circle table
    for b in (1, 2, 3, 4):
        c1 = oracle.angle_codebook(1, b)
        D = 2 * pi / 2 ** b
        assert np.allclose(c1.centroids, (np.arange(2 ** b) + 0.5) * D)
        assert np.allclose(c1.thresholds, np.arange(1, 2 ** b) * D)
        assert c1.distortion() == pytest.approx(D * D / 12, rel=1e-9)


@pytest.mark.parametrize("level", [2, 3, 4, 6])
@pytest.mark.parametrize("bits", [2, 3])
def test_lloyd_conditions_by_sampling(level, bits):
    # centroids are the cell means of the law (sampled by another route: psi = asin(sqrt(Beta)))
    # and thresholds the centroid midpoints; the table is symmetric about pi/4
    cb = oracle.angle_codebook(level, bits)
    k = oracle.angle_dof(level)
    g = np.random.default_rng(1000 + 10 * level + bits)
    psi = np.arcsin(np.sqrt(g.beta(k / 2, k / 2, size=400000)))
    idx = cb.codes(psi)
    for j, c in enumerate(cb.centroids):
        cell = psi[idx == j]
        assert abs(cell.mean() - c) < 5 * cell.std() / np.sqrt(cell.size)
    assert np.allclose(cb.thresholds, (cb.centroids[1:] + cb.centroids[:-1]) / 2)
    assert np.allclose(cb.centroids + cb.centroids[::-1], pi / 2, atol=1e-12)


def test_codes_are_the_nearest_centroid():
    g = np.random.default_rng(3)
    for level in (1, 2, 5):
        for bits in (1, 2, 3):
            cb = oracle.angle_codebook(level, bits)
            hi = 2 * pi if level == 1 else pi / 2
            psi = g.uniform(0, hi, size=5000)
            dist = np.abs(psi[:, None] - cb.centroids[None, :])
            if level == 1:
                dist = np.minimum(dist, 2 * pi - dist)   # on the circle
            assert np.array_equal(cb.codes(psi), np.argmin(dist, axis=1))


def test_distortion_falls_with_bits_and_matches_the_levels():
    # D = E|x - x_hat|^2 / |x|^2 by Monte Carlo falls with b, and at b = 4 it is small
    d, n = 64, 3000
    Pi, _ = rng.method_matrices(5, d, 1)
    X = rng.gaussian_stream(6, n * d).reshape(n, d)
    prev = np.inf
    for b in (1, 2, 3, 4):
        pcb = oracle.polar_codebook(d, b)
        z = oracle.polar_quantize(X, Pi, pcb)
        Xh = oracle.polar_dequantize(z.codes, z.r16, Pi, pcb)
        D = np.mean(np.sum((X - Xh) ** 2, axis=1) / np.sum(X ** 2, axis=1))
        assert D < prev
        prev = D
    assert prev < 0.02


def test_estimator_is_unbiased_over_seeds():
    d, n, b = 16, 4000, 2
    pcb = oracle.polar_codebook(d, b)
    x, q = rng.gaussian_stream(2001, d), rng.gaussian_stream(2002, d)
    err = np.empty(n)
    for s in range(n):
        Pi, S = rng.method_matrices(50_000 + s, d, d)
        z = oracle.polar_quantize(x[None], Pi, pcb, S)
        err[s] = oracle.polar_estimate(q, z, Pi, pcb, S)[0] - q @ x
    assert abs(err.mean()) < 3 * err.std() / np.sqrt(n)


def test_mse_only_estimate_is_the_inner_product_with_the_reconstruction():
    d = 32
    pcb = oracle.polar_codebook(d, 3)
    Pi, _ = rng.method_matrices(8, d, 1)
    X = rng.gaussian_stream(9, 10 * d).reshape(10, d)
    q = rng.gaussian_stream(10, d)
    z = oracle.polar_quantize(X, Pi, pcb)
    brute = np.array([q @ xh for xh in oracle.polar_dequantize(z.codes, z.r16, Pi, pcb)])
    assert np.allclose(oracle.polar_estimate(q, z, Pi, pcb), brute, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("d,b", [(128, 3), (128, 2), (64, 4), (8, 1)])
def test_packing_layout(d, b):
    g = np.random.default_rng(11)
    codes = g.integers(0, 2 ** b, size=(6, d - 1))
    words = oracle.pack_polar(codes, b)
    assert words.shape == (6, ((d - 1) * b + 31) // 32) and words.dtype == np.uint32
    assert np.array_equal(oracle.unpack_polar(words, d, b), codes)
    for r, a in [(0, 0), (2, d // 2), (5, d - 2), (3, 10 % (d - 1))]:
        for i in range(b):
            t = a * b + i
            assert (int(words[r, t // 32]) >> (t % 32)) & 1 == (codes[r, a] >> i) & 1
