"""Oracle for the recursive polar-angle encoder (the PolarQuant representation the pages describe).

TEST INFRASTRUCTURE, like the rest of this package: only tests/, smoke() and bench.py's CPU legs
use it.  Plain float64 numpy; scipy's regularised incomplete beta and adaptive quadrature serve as
single library steps.

What the pages fix (by title and section):

* csdn tutorial, section "将笛卡尔积坐标转为极坐标": a d-dimensional vector becomes its Euclidean
  length r (kept at higher precision, FP16) plus d - 1 angles that give its direction on the unit
  sphere; the angles are concentrated and are stored at low precision (2 or 3 bits).
* csdn tutorial, section "TurboQuant原理剖析": r at 16 bits, the angles at 2 bits (3 bits in total
  with the 1 QJL bit) or 3 bits (4 in total); then 1 sign bit per dimension of the Gaussian
  projection of the residual (QJL).
* freelamp article, section "技术突破：极坐标量化": a random orthogonal rotation first; after it the
  angle components follow a known analytic law; a recursive polar transform reduces the vector to
  one radius and a series of angles; no per-block scaling constants.
* csdn tutorial, section "PolarQuant": the 4-dimensional worked example, where the rotation maps the
  column vector to [5, 5, 5, 5]^T.

Readings (where the pages leave a step open):

1. The recursion pairs neighbours: level 1 takes (y_2i, y_2i+1) to a radius and an angle, level l
   pairs the radii of level l - 1 the same way, until one radius is left (d a power of two).  That
   gives d/2 + d/4 + ... + 1 = d - 1 angles, the count the pages give for d = 4096.
2. A level-1 angle is atan2(y_2i+1, y_2i) taken in [0, 2 pi); a level-l angle (l >= 2) is
   atan2(right radius, left radius) in [0, pi/2].
3. The analytic law after the rotation: y / |y| is uniform on the sphere, so the level-1 angles are
   uniform on the circle and a level-l angle has density proportional to (sin psi cos psi)^(k-1)
   on [0, pi/2], k = 2^(l-1) (the two child radii are independent chi variables with k degrees of
   freedom each, so sin^2 psi ~ Beta(k/2, k/2)).
4. Every angle gets the same bit width b; each level has its own Lloyd-Max table for its law.  On
   the circle (level 1) the table is the uniform one: cells [j D, (j + 1) D), centroids (j + 1/2) D,
   D = 2 pi / 2^b.
5. r16 = fp16(|x|) (= |y|); the reconstruction is x_hat = Pi^T y_hat with y_hat rebuilt top-down
   from r16 and the angle centroids; the QJL stage and the estimator are the main path's, on the
   residual x - x_hat: est = <Pi q, y_hat> + rnorm16 sqrt(pi/2)/m <S q, 2 sigma - 1>.
6. Packed layout: the d - 1 codes in angle order (level 1 left to right, then level 2, ...) as
   consecutive b-bit fields of one little-endian bit stream: code a holds stream bits a*b .. a*b+b-1,
   stream bit t is bit t % 32 of word t / 32; ceil((d - 1) b / 32) words per vector.
"""
from __future__ import annotations

from dataclasses import dataclass
from math import pi, sqrt
from typing import List, Optional

import numpy as np
from scipy import integrate, special

from .turboquant import QJL_CONST, fp16_round


def _levels(d: int) -> int:
    L = int(d).bit_length() - 1
    if d < 2 or (1 << L) != d:
        raise ValueError("the recursive polar transform needs d a power of two >= 2")
    return L


# ----------------------------------------------------------------------------- transform

def polar_forward(Y: np.ndarray):
    """Reading 1-2: rows of Y [n, d] -> (r [n], angles: list over levels of [n, d / 2^l],
    radii: list over levels of [n, d / 2^l] (the radius each angle was taken at))."""
    Y = np.asarray(Y, dtype=np.float64)
    _levels(Y.shape[-1])
    angles, radii = [], []
    cur = Y
    level = 1
    while cur.shape[-1] > 1:
        a, b = cur[..., 0::2], cur[..., 1::2]
        rad = np.sqrt(a * a + b * b)
        ang = np.arctan2(b, a)
        if level == 1:
            ang = np.where(ang < 0.0, ang + 2.0 * pi, ang)   # [0, 2 pi)
            ang = np.where(ang >= 2.0 * pi, 0.0, ang)
        angles.append(ang)
        radii.append(rad)
        cur = rad
        level += 1
    return cur[..., 0], angles, radii


def polar_inverse(r: np.ndarray, angles: List[np.ndarray]) -> np.ndarray:
    """Top-down rebuild: a node of radius rho and angle psi has children rho cos psi (left) and
    rho sin psi (right); the level-1 children are the coordinates."""
    cur = np.asarray(r, dtype=np.float64)[..., None]
    for ang in reversed(angles):
        ang = np.asarray(ang, dtype=np.float64)
        out = np.empty(cur.shape[:-1] + (2 * cur.shape[-1],))
        out[..., 0::2] = cur * np.cos(ang)
        out[..., 1::2] = cur * np.sin(ang)
        cur = out
    return cur


# ----------------------------------------------------------------------------- angle laws and tables

def angle_dof(level: int) -> int:
    """Degrees of freedom k of each child radius of a level-l angle (reading 3): k = 2^(l-1)."""
    return 1 << (level - 1)


def angle_pdf(psi: np.ndarray, level: int) -> np.ndarray:
    """Density of a level-l angle.  Level 1: 1 / (2 pi) on [0, 2 pi).  Level l >= 2:
    2 (sin psi cos psi)^(k-1) / B(k/2, k/2) on [0, pi/2] (sin^2 psi ~ Beta(k/2, k/2))."""
    psi = np.asarray(psi, dtype=np.float64)
    if level == 1:
        return np.where((psi >= 0) & (psi < 2 * pi), 1.0 / (2 * pi), 0.0)
    k = angle_dof(level)
    s = np.clip(np.sin(psi) * np.cos(psi), 0.0, None)
    inside = (psi >= 0) & (psi <= pi / 2)
    return np.where(inside, 2.0 * s ** (k - 1) / special.beta(k / 2, k / 2), 0.0)


def angle_cdf(psi: np.ndarray, level: int) -> np.ndarray:
    """P(angle <= psi): psi / (2 pi) at level 1, I_{sin^2 psi}(k/2, k/2) at level l >= 2."""
    psi = np.asarray(psi, dtype=np.float64)
    if level == 1:
        return np.clip(psi / (2 * pi), 0.0, 1.0)
    k = angle_dof(level)
    p = np.clip(psi, 0.0, pi / 2)
    return special.betainc(k / 2, k / 2, np.sin(p) ** 2)


_GL_X, _GL_W = np.polynomial.legendre.leggauss(96)


def _first_moment(a: np.ndarray, b: np.ndarray, level: int) -> np.ndarray:
    """int_a^b psi f(psi) dpsi per cell, 96-point Gauss-Legendre on each cell."""
    half, mid = (b - a) / 2.0, (b + a) / 2.0
    psi = mid[:, None] + half[:, None] * _GL_X[None, :]
    return half * np.sum(_GL_W[None, :] * psi * angle_pdf(psi, level), axis=1)


@dataclass
class AngleCodebook:
    """Lloyd-Max table of one level: 2^bits centroids ascending, 2^bits - 1 inner thresholds."""

    level: int
    bits: int
    centroids: np.ndarray
    thresholds: np.ndarray

    def codes(self, psi: np.ndarray) -> np.ndarray:
        """Index of the cell holding psi = number of thresholds strictly below it."""
        return np.searchsorted(self.thresholds, np.asarray(psi, dtype=np.float64), side="left").astype(np.int64)

    def distortion(self) -> float:
        """E (psi - c(psi))^2 under the level's law, by quadrature cell by cell."""
        lo = 0.0
        hi = 2 * pi if self.level == 1 else pi / 2
        edges = np.concatenate([[lo], self.thresholds, [hi]])
        tot = 0.0
        for j, c in enumerate(self.centroids):
            tot += integrate.quad(lambda t: (t - c) ** 2 * float(angle_pdf(np.array(t), self.level)),
                                  edges[j], edges[j + 1], limit=200, epsabs=1e-15, epsrel=1e-12)[0]
        return tot


def angle_codebook(level: int, bits: int, tol: float = 1e-14, max_iter: int = 100000) -> AngleCodebook:
    """Reading 4: the uniform circle table at level 1; the Lloyd iteration (thresholds at the
    midpoints, centroids at the cell means: mass from the closed-form CDF, first moment by
    quadrature) from the quantile start at levels >= 2."""
    n = 1 << bits
    if level == 1:
        D = 2 * pi / n
        return AngleCodebook(level, bits, (np.arange(n) + 0.5) * D, np.arange(1, n) * D)
    k = angle_dof(level)
    p = (np.arange(n) + 0.5) / n
    c = np.arcsin(np.sqrt(special.betaincinv(k / 2, k / 2, p)))
    for _ in range(max_iter):
        t = (c[:-1] + c[1:]) / 2.0
        edges = np.concatenate([[0.0], t, [pi / 2]])
        mass = np.diff(angle_cdf(edges, level))
        new = _first_moment(edges[:-1], edges[1:], level) / mass
        done = np.max(np.abs(new - c)) < tol
        c = new
        if done:
            break
    return AngleCodebook(level, bits, c, (c[:-1] + c[1:]) / 2.0)


@dataclass
class PolarCodebook:
    """The per-level tables of a d-dimensional polar encoder with b bits per angle."""

    d: int
    bits: int
    levels: List[AngleCodebook]

    @property
    def n_angles(self) -> int:
        return self.d - 1


def polar_codebook(d: int, bits: int) -> PolarCodebook:
    L = _levels(d)
    return PolarCodebook(d, bits, [angle_codebook(l, bits) for l in range(1, L + 1)])


# ----------------------------------------------------------------------------- encoder and estimator

@dataclass
class PolarQuantized:
    """Codes of n vectors: codes [n, d - 1] (angle order of reading 6), r16 [n], and for the QJL
    stage signs [n, m] (bool) and rnorm16 [n]."""

    codes: np.ndarray
    r16: np.ndarray
    signs: Optional[np.ndarray] = None
    rnorm16: Optional[np.ndarray] = None


def _split_levels(flat: np.ndarray, d: int) -> List[np.ndarray]:
    out, a, w = [], 0, d // 2
    while w >= 1:
        out.append(flat[..., a:a + w])
        a += w
        w //= 2
    return out


def polar_codes(Y: np.ndarray, pcb: PolarCodebook) -> np.ndarray:
    """Codes [n, d - 1] of the rotated rows Y: each angle's cell in its level's table."""
    _, angles, _ = polar_forward(Y)
    return np.concatenate([cb.codes(a) for cb, a in zip(pcb.levels, angles)], axis=-1)


def polar_rebuild(codes: np.ndarray, r16: np.ndarray, pcb: PolarCodebook) -> np.ndarray:
    """y_hat [n, d] from the codes and the stored radius (reading 5)."""
    levels = _split_levels(np.asarray(codes), pcb.d)
    return polar_inverse(r16, [cb.centroids[c] for cb, c in zip(pcb.levels, levels)])


def polar_dequantize(codes: np.ndarray, r16: np.ndarray, Pi: np.ndarray, pcb: PolarCodebook) -> np.ndarray:
    """x_hat = Pi^T y_hat (row form y_hat @ Pi)."""
    return polar_rebuild(codes, r16, pcb) @ Pi


def polar_quantize(X: np.ndarray, Pi: np.ndarray, pcb: PolarCodebook, S: Optional[np.ndarray] = None) -> PolarQuantized:
    """Rotate, recursive polar transform, per-level angle codes, fp16 radius; with S the QJL
    signs of S (x - x_hat) and the fp16 residual norm."""
    X = np.asarray(X, dtype=np.float64)
    Y = X @ Pi.T
    codes = polar_codes(Y, pcb)
    r16 = fp16_round(np.linalg.norm(X, axis=-1))
    if S is None:
        return PolarQuantized(codes=codes, r16=r16)
    R = X - polar_dequantize(codes, r16, Pi, pcb)
    return PolarQuantized(codes=codes, r16=r16, signs=(R @ S.T) > 0.0,
                          rnorm16=fp16_round(np.linalg.norm(R, axis=-1)))


def polar_estimate(q: np.ndarray, z: PolarQuantized, Pi: np.ndarray, pcb: PolarCodebook,
                   S: Optional[np.ndarray] = None) -> np.ndarray:
    """est(q, x) = <Pi q, y_hat> (+ rnorm16 sqrt(pi/2)/m <S q, 2 sigma - 1>) for every coded row."""
    q = np.asarray(q, dtype=np.float64)
    est = polar_rebuild(z.codes, z.r16, pcb) @ (Pi @ q)
    if S is None:
        return est
    sigma = 2.0 * z.signs.astype(np.float64) - 1.0
    return est + z.rnorm16 * (QJL_CONST / S.shape[0]) * (sigma @ (S @ q))


# ----------------------------------------------------------------------------- packing

def polar_words(d: int, bits: int) -> int:
    return ((d - 1) * bits + 31) // 32


def pack_polar(codes: np.ndarray, bits: int) -> np.ndarray:
    """Reading 6: codes [n, d - 1] -> words [n, ceil((d - 1) bits / 32)] uint32."""
    codes = np.asarray(codes, dtype=np.int64)
    n, na = codes.shape
    stream = ((codes[:, :, None] >> np.arange(bits)[None, None, :]) & 1).reshape(n, na * bits)
    W = polar_words(na + 1, bits)
    padded = np.zeros((n, 32 * W), dtype=np.uint64)
    padded[:, :na * bits] = stream
    return (padded.reshape(n, W, 32) << np.arange(32, dtype=np.uint64)).sum(axis=2).astype(np.uint32)


def unpack_polar(words: np.ndarray, d: int, bits: int) -> np.ndarray:
    words = np.asarray(words, dtype=np.uint32).astype(np.uint64)
    n = words.shape[0]
    stream = ((words[:, :, None] >> np.arange(32, dtype=np.uint64)) & 1).reshape(n, -1)[:, :(d - 1) * bits]
    return (stream.reshape(n, d - 1, bits).astype(np.int64) << np.arange(bits)).sum(axis=2)
