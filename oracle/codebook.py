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
from scipy.linalg import solve_banded
from scipy.special import betaincc, betainccinv, ndtri


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


# Stop rule of the Newton solve: a further Lloyd step moves no centroid by more than this.  It is
# the rounding floor of the step itself: a cell's probability is a difference of incomplete-beta
# values of size ~1/2 (absolute error ~1e-16), i.e. ~1e-14 relative for a cell of probability
# 1/256, and the cell mean inherits that.
NEWTON_TOL = 5e-14


def _cells(c: np.ndarray, d: float):
    """Midpoint thresholds of the centroids c and, per cell, (lo, hi, P_k, E[T | cell])."""
    t = 0.5 * (c[:-1] + c[1:])
    lo = np.concatenate(([-1.0], t))
    hi = np.concatenate((t, [1.0]))
    p = sphere_cell_prob(lo, hi, d)
    return t, lo, hi, p, sphere_cell_first_moment(lo, hi, d) / p


def _sphere_quantiles(probs: np.ndarray, d: float) -> np.ndarray:
    """t with P(T < t) = prob for the density proportional to (1 - t^2)^((d-3)/2), d > 1 real:
    T^2 ~ Beta(1/2, (d-1)/2), so the inverse of the regularised incomplete beta gives |t|."""
    probs = np.asarray(probs, dtype=np.float64)
    upper = np.where(probs < 0.5, probs, 1.0 - probs)          # P(T > |t|) = upper
    a = np.sqrt(betainccinv(0.5, 0.5 * (d - 1), 2.0 * upper))
    return np.where(probs < 0.5, -a, a)


def _newton_lloyd(c: np.ndarray, d: int, tol: float, max_iter: int = 200) -> np.ndarray:
    """Solves the Lloyd-Max conditions c_k = E[T | t_(k-1) < T < t_k], t_k = (c_k + c_(k+1))/2
    by Newton's method on F(c) = g(c) - c, g one Lloyd step, until one more Lloyd step would move
    no centroid by more than ``tol`` (the rounding level of the step itself).  With
    A_k = f(lo_k)(g_k - lo_k)/P_k and B_k = f(hi_k)(hi_k - g_k)/P_k (the derivatives of the cell
    mean in its edges, which move by 1/2 with each neighbouring centroid), the Jacobian of c - g is
    tridiagonal:
        row k:  -A_k/2 at c_(k-1),  1 - (A_k + B_k)/2 at c_k,  -B_k/2 at c_(k+1).
    A step that would break the ordering of the centroids is halved."""
    L = len(c)
    for _ in range(max_iter):
        _, lo, hi, p, g = _cells(c, d)
        if np.max(np.abs(g - c)) <= tol:
            return c
        A = np.where(np.arange(L) > 0, sphere_marginal_pdf(lo, d) * (g - lo) / p, 0.0)
        B = np.where(np.arange(L) < L - 1, sphere_marginal_pdf(hi, d) * (hi - g) / p, 0.0)
        ab = np.zeros((3, L))
        ab[0, 1:] = -0.5 * B[:-1]          # upper diagonal: row k, column k + 1
        ab[1] = 1.0 - 0.5 * (A + B)
        ab[2, :-1] = -0.5 * A[1:]          # lower diagonal: row k, column k - 1
        step = solve_banded((1, 1), ab, g - c)
        while True:
            c_new = c + step
            if np.all(np.diff(c_new) > 0) and -1.0 < c_new[0] and c_new[-1] < 1.0:
                break
            step = 0.5 * step
        c = c_new
    raise RuntimeError("Newton iteration on the Lloyd-Max conditions did not converge")


def sphere_codebook(d: int, bits: int, tol: float = 4e-16, max_iter: int = 200000) -> Codebook:
    """Lloyd-Max quantizer with 2**bits levels for the density f_d: the fixed point of
    thresholds t_k = (c_k + c_{k+1}) / 2 and centroids c_k = E[T | t_{k-1} < T < t_k]
    (t_{-1} = -1, t_{L-1} = 1), which is unique since f_d is log-concave.

    1 to 4 bits: the Lloyd iteration itself, started at the levels of the N(0, 1/d) quantiles
    at (k + 1/2) / L, stopped when no centroid moves by more than ``tol`` (rounding level: the
    fixed point is reached to ~1e-16, not just slowed down).
    5 to 8 bits: one Lloyd step contracts the error by only ~1 - O(1/L^2) there, so the same
    fixed point is solved for by Newton's method (``_newton_lloyd``), started at the
    high-resolution optimum (centroid density proportional to f_d^(1/3), i.e. the quantiles at
    (k + 1/2) / L of the same family with (d - 3)/2 replaced by (d - 3)/6) and stopped on the
    residual rule at the rounding floor of a Lloyd step (``NEWTON_TOL``).
    Finally the table is symmetrised (f_d is even).
    """
    if d < 3:
        raise ValueError("the sphere-marginal codebook needs d >= 3")
    if not 1 <= bits <= 8:
        raise ValueError("bits must be in 1..8")
    L = 1 << bits
    if bits <= 4:
        c = ndtri((np.arange(L) + 0.5) / L) / sqrt(d)
        for _ in range(max_iter):
            _, _, _, _, c_new = _cells(c, d)
            moved = np.max(np.abs(c_new - c))
            c = c_new
            if moved < tol:
                break
        else:
            raise RuntimeError("Lloyd iteration did not converge")
    else:
        c = _newton_lloyd(_sphere_quantiles((np.arange(L) + 0.5) / L, (d + 6.0) / 3.0), d, NEWTON_TOL)
    c = 0.5 * (c - c[::-1])
    t = 0.5 * (c[:-1] + c[1:])
    if L % 2 == 0:
        t[L // 2 - 1] = 0.0
    lo = np.concatenate(([-1.0], t))
    hi = np.concatenate((t, [1.0]))
    return Codebook(d=d, bits=bits, centroids=c, thresholds=t, cell_prob=sphere_cell_prob(lo, hi, d))
