"""Seeded random matrices of the method: the rotation Pi and the JL projection S.

Test infrastructure only (see the package docstring).

The pages fix only the laws: a random orthogonal rotation applied before
quantization ([freelamp PQ]; [juejin §2]; [csdn PolarQuant]) and a Gaussian
JL projection of the residual ([csdn QJL-1]).  Any fixed generator is correct,
and parity never depends on it because the GPU library accepts the matrices
as data.  The generator below is the one the library also implements (in its
own C++), so that ``tq_init(seed, ...)`` can be checked against it:

* splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): state advances by the golden-ratio increment
  0x9E3779B97F4A7C15 and each output is the state passed through the
  variant-13 finaliser (xor-shift 30, multiply 0xBF58476D1CE4E5B9, xor-shift 27,
  multiply 0x94D049BB133111EB, xor-shift 31).  Output k (k = 0, 1, ...) uses
  state seed + (k + 1) * increment.
* A uniform in (0, 1]: u = ((z >> 11) + 1) * 2^-53.
* Box-Muller: the pair (u1, u2) = (uniform 2k, uniform 2k+1) gives
  g_2k = sqrt(-2 ln u1) cos(2 pi u2) and g_2k+1 = sqrt(-2 ln u1) sin(2 pi u2).
* S (m x d) takes normals 0 .. m*d-1 row-major; the Gaussian G (d x d) for Pi
  takes the next d*d normals row-major.
* Pi = Q diag(sign(diag R)) where G = QR (Householder); the sign fix makes Pi
  Haar-distributed (Mezzadri, "How to generate random matrices from the
  classical compact groups", Notices AMS 2007).
"""

from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64_stream(seed: int, count: int, start: int = 0) -> np.ndarray:
    """Outputs start .. start+count-1 of splitmix64 seeded with ``seed`` (uint64)."""
    k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + k * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def gaussian_stream(seed: int, count: int) -> np.ndarray:
    """The first ``count`` standard normals of the Box-Muller stream (float64)."""
    pairs = (count + 1) // 2
    z = splitmix64_stream(seed, 2 * pairs)
    u = ((z >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    th = 2.0 * np.pi * u2
    g = np.empty(2 * pairs, dtype=np.float64)
    g[0::2] = r * np.cos(th)
    g[1::2] = r * np.sin(th)
    return g[:count]


def haar_rotation(G: np.ndarray) -> np.ndarray:
    """Pi = Q diag(sign(diag R)) for G = QR: a Haar-random orthogonal matrix."""
    Q, R = np.linalg.qr(G)
    s = np.sign(np.diag(R))
    s[s == 0] = 1.0
    return Q * s[None, :]


def jl_matrix(seed: int, m: int, d: int) -> np.ndarray:
    """S with i.i.d. N(0, 1) entries, m x d ([csdn QJL-1]: Gaussian JL projection)."""
    return gaussian_stream(seed, m * d).reshape(m, d)


def method_matrices(seed: int, d: int, m: int) -> tuple[np.ndarray, np.ndarray]:
    """(Pi, S) for ``seed``, float64, drawn from one stream as the module docstring says."""
    g = gaussian_stream(seed, m * d + d * d)
    S = g[: m * d].reshape(m, d)
    G = g[m * d:].reshape(d, d)
    return haar_rotation(G), S
