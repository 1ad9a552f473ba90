"""Data-oblivious scalar codebook for the rotated coordinates (Lloyd-Max).

Test infrastructure only (see the package docstring).

What the pages fix: after the random rotation the coordinates follow a
concentrated, predictable law ([freelamp PQ]; [juejin §2]); the quantizer maps
each coordinate to the nearest allowed discrete value ([csdn QJL], opening
paragraph); the centroids sit where probability is higher and are precomputed
once for all tokens and layers ([nonnda 3.2], [nonnda 3.4]); no per-block
constants are stored ([freelamp PQ]).

Reading taken here (the pages print neither the density nor the centroids):
after a Haar rotation, Pi x / ||x|| is exactly uniform on the unit sphere of
R^d for every x != 0, so one coordinate T has the density

    f_d(t) = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)) * (1 - t^2)^((d-3)/2),  |t| <= 1,

and the MSE-optimal b-bit scalar quantizer for T is the Lloyd-Max quantizer of
f_d.  It is computed here by the Lloyd iteration (thresholds at midpoints,
centroids at conditional means) with the cell integrals in closed form:

* P(a < T < b) from the regularised incomplete beta function, since T^2 follows
  Beta(1/2, (d-1)/2);
* the first moment from d/dt (1 - t^2)^((d-1)/2) = -(d-1) t (1 - t^2)^((d-3)/2).

The GPU library computes its own table by a different route (Gauss-Legendre
quadrature of f_d in C++); the tests compare the two.
"""

from __future__ import annotations

from dataclasses import dataclass
from math import lgamma, log, exp, pi, sqrt

import numpy as np
from scipy.special import betaincc, ndtri


def _log_norm_const(d: int) -> float:
    return lgamma(d / 2.0) - 0.5 * log(pi) - lgamma((d - 1) / 2.0)


def sphere_marginal_pdf(t: np.ndarray, d: int) -> np.ndarray:
    """f_d(t): density of one coordinate of a uniform unit vector in R^d (d >= 3)."""
    t = np.asarray(t, dtype=np.float64)
    out = np.zeros_like(t)
    inside = np.abs(t) < 1.0
    out[inside] = np.exp(_log_norm_const(d) + 0.5 * (d - 3) * np.log1p(-t[inside] ** 2))
    return out


def _upper_tail(t: np.ndarray, d: int) -> np.ndarray:
    """P(T > t) for t >= 0: half of P(T^2 > t^2), T^2 ~ Beta(1/2, (d-1)/2)."""
    return 0.5 * betaincc(0.5, 0.5 * (d - 1), np.asarray(t, dtype=np.float64) ** 2)


def _cdf(t: np.ndarray, d: int) -> np.ndarray:
    t = np.asarray(t, dtype=np.float64)
    return np.where(t >= 0, 1.0 - _upper_tail(np.abs(t), d), _upper_tail(np.abs(t), d))


def sphere_cell_prob(a: np.ndarray, b: np.ndarray, d: int) -> np.ndarray:
    """P(a < T < b) for -1 <= a <= b <= 1, avoiding cancellation in either tail."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    pos = a >= 0
    neg = b <= 0
    mid = ~(pos | neg)
    out = np.empty(np.broadcast(a, b).shape)
    out[pos] = _upper_tail(a[pos], d) - _upper_tail(b[pos], d)
    out[neg] = _upper_tail(-b[neg], d) - _upper_tail(-a[neg], d)
    out[mid] = 1.0 - _upper_tail(-a[mid], d) - _upper_tail(b[mid], d)
    return out


def sphere_cell_first_moment(a: np.ndarray, b: np.ndarray, d: int) -> np.ndarray:
    """Integral of t f_d(t) over (a, b), in closed form."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    k = exp(_log_norm_const(d)) / (d - 1)

    def g(t):
        t = np.atleast_1d(t)
        out = np.zeros_like(t)
        inside = np.abs(t) < 1.0
        out[inside] = np.exp(0.5 * (d - 1) * np.log1p(-t[inside] ** 2))
        return out

    return k * (g(a) - g(b))


@dataclass
class Codebook:
    """Centroids c[0..L-1] ascending (index 0 the most negative) and L-1 thresholds."""

    d: int
    bits: int
    centroids: np.ndarray
    thresholds: np.ndarray
    cell_prob: np.ndarray

    @property
    def levels(self) -> int:
        return len(self.centroids)

    def distortion(self) -> float:
        """Expected ||u - c[idx]||^2 for u uniform on the sphere: d * E[(T - c(T))^2].

        With the centroid condition E[T c(T)] = E[c(T)^2], this is 1 - d * sum_k P_k c_k^2.
        """
        return float(1.0 - self.d * np.sum(self.cell_prob * self.centroids ** 2))


def sphere_codebook(d: int, bits: int, tol: float = 4e-16, max_iter: int = 200000) -> Codebook:
    """Lloyd-Max quantizer with 2**bits levels for the density f_d.

    Start: the levels of the N(0, 1/d) quantiles at (k + 1/2) / L (a start only).
    Step:  thresholds t_k = (c_k + c_{k+1}) / 2; centroids c_k = E[T | t_{k-1} < T < t_k]
           with t_{-1} = -1 and t_{L-1} = 1.
    Stop:  when no centroid moves by more than ``tol`` (rounding level: the fixed point is
           reached to ~1e-16, not just slowed down); then symmetrise (f_d is even).
    """
    if d < 3:
        raise ValueError("the sphere-marginal codebook needs d >= 3")
    if not 1 <= bits <= 8:
        raise ValueError("bits must be in 1..8")
    L = 1 << bits
    c = ndtri((np.arange(L) + 0.5) / L) / sqrt(d)
    for _ in range(max_iter):
        t = 0.5 * (c[:-1] + c[1:])
        lo = np.concatenate(([-1.0], t))
        hi = np.concatenate((t, [1.0]))
        p = sphere_cell_prob(lo, hi, d)
        c_new = sphere_cell_first_moment(lo, hi, d) / p
        moved = np.max(np.abs(c_new - c))
        c = c_new
        if moved < tol:
            break
    else:
        raise RuntimeError("Lloyd iteration did not converge")
    c = 0.5 * (c - c[::-1])
    t = 0.5 * (c[:-1] + c[1:])
    if L % 2 == 0:
        t[L // 2 - 1] = 0.0
    lo = np.concatenate(([-1.0], t))
    hi = np.concatenate((t, [1.0]))
    return Codebook(d=d, bits=bits, centroids=c, thresholds=t, cell_prob=sphere_cell_prob(lo, hi, d))
