"""Pins for the sphere-marginal Lloyd-Max codebook."""
from math import exp, lgamma, pi, sqrt

import numpy as np
import pytest

from oracle.codebook import sphere_codebook, sphere_marginal_pdf, sphere_cell_prob
from conftest import read_golden


def _gl_integral(f, a, b, n=400):
    x, w = np.polynomial.legendre.leggauss(n)
    t = 0.5 * (b - a) * x + 0.5 * (b + a)
    return 0.5 * (b - a) * np.sum(w * f(t))


@pytest.mark.parametrize("d", [3, 16, 128, 200])
def test_density_integrates_to_one(d):
    total = sum(_gl_integral(lambda t: sphere_marginal_pdf(t, d), a, a + 0.25) for a in np.arange(-1, 1, 0.25))
    assert abs(total - 1.0) < 1e-12
    # second moment of one coordinate of a unit vector is 1/d
    m2 = sum(_gl_integral(lambda t: t * t * sphere_marginal_pdf(t, d), a, a + 0.25) for a in np.arange(-1, 1, 0.25))
    assert abs(m2 - 1.0 / d) < 1e-12


@pytest.mark.parametrize("d,c1,D1", [(128, 0.0706616, 0.360889), (200, 0.0564895, 0.361787)])
def test_one_bit_closed_form(d, c1, D1):
    cb = sphere_codebook(d, 1)
    exact = exp(lgamma(d / 2) - lgamma((d + 1) / 2)) / sqrt(pi)   # E|T|
    assert abs(cb.centroids[1] - exact) < 1e-14
    assert abs(cb.centroids[0] + exact) < 1e-14
    assert cb.thresholds[0] == 0.0
    assert abs(cb.centroids[1] - c1) < 5e-8
    assert abs(cb.distortion() - (1 - d * exact ** 2)) < 1e-12
    assert abs(cb.distortion() - D1) < 5e-7


@pytest.mark.parametrize("d", [16, 128, 200])
@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 8])
def test_lloyd_conditions_by_independent_quadrature(d, bits):
    cb = sphere_codebook(d, bits)
    c, t = cb.centroids, cb.thresholds
    L = len(c)
    assert L == 2 ** bits and len(t) == L - 1
    assert np.all(np.diff(c) > 0) and np.all(np.diff(t) > 0)
    assert np.array_equal(c, -c[::-1])                      # symmetric table
    assert np.allclose(t, 0.5 * (c[:-1] + c[1:]), atol=1e-15, rtol=0)   # midpoint condition
    edges = np.concatenate(([-1.0], t, [1.0]))
    for k in range(L):
        a, b = edges[k], edges[k + 1]
        # the density is negligible beyond 12 standard deviations; keep quadrature nodes there
        a, b = max(a, -12 / sqrt(d)), min(b, 12 / sqrt(d))
        p = _gl_integral(lambda s: sphere_marginal_pdf(s, d), a, b)
        mu = _gl_integral(lambda s: s * sphere_marginal_pdf(s, d), a, b)
        assert abs(mu / p - c[k]) < 1e-12                   # centroid condition
        assert abs(p - cb.cell_prob[k]) < 1e-12


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_gaussian_limit_matches_max_1960(bits):
    g = read_golden("gaussian_lloyd_max.txt")
    d = 10 ** 6
    cb = sphere_codebook(d, bits)
    pos = sqrt(d) * cb.centroids[len(cb.centroids) // 2:]
    assert np.allclose(pos, g["levels_%d" % bits], rtol=0, atol=6e-4)
    assert abs(cb.distortion() - g["mse_%d" % bits][0]) < 1.5e-4


@pytest.mark.parametrize("d", [16, 128])
def test_distortion_falls_with_bits(d):
    D = [sphere_codebook(d, b).distortion() for b in range(1, 9)]
    assert all(D[i + 1] < D[i] for i in range(7))
    # rate-distortion sanity: each extra bit buys at least a factor ~3 (the Gaussian limit is ~3.1-3.6,
    # tending to 4 at high rate)
    assert all(4.0 > D[i] / D[i + 1] > 2.9 for i in range(7))


def test_high_rate_limit_panter_dite():
    # High-resolution theory (Panter and Dite, 1951): the b-bit Lloyd-Max distortion of a unit
    # Gaussian behaves as (pi sqrt(3) / 2) 4^-b.  In the d -> infinity limit of the sphere marginal
    # (sqrt(d) T -> N(0, 1)) the solved tables approach that constant from below as b grows.
    C = pi * sqrt(3.0) / 2.0
    d = 10 ** 6
    r = [sphere_codebook(d, b).distortion() * 4 ** b for b in (5, 6, 7, 8)]
    assert all(r[i] < r[i + 1] < C for i in range(3))
    assert abs(r[-1] / C - 1.0) < 0.015


def test_cell_probabilities_sum_to_one():
    cb = sphere_codebook(128, 3)
    assert abs(cb.cell_prob.sum() - 1.0) < 1e-14
    assert abs(sphere_cell_prob(np.array([-1.0]), np.array([1.0]), 128)[0] - 1.0) < 1e-15
