"""The TurboQuant hot path, written out plainly in float64.

Test infrastructure only (see the package docstring for the citation legend).

Steps, in the pages' order:

1. PolarQuant stage ([juejin §2]; [freelamp PQ]; [csdn PolarQuant]; [csdn polar]):
   n = ||x||_2 kept as fp16; y = Pi x; u = y / n; each u_j is coded by the
   nearest centroid of the precomputed table (index = number of thresholds
   below u_j, so a value exactly on a threshold takes the lower index).
2. QJL stage ([csdn QJL-1], [csdn QJL-2]; [juejin §2]): the residual
   r = x - x_hat, where x_hat = n16 * Pi^T c[idx] is what the PolarQuant codes
   reconstruct; the signs of S r are kept as bits (> 0 -> 1; reading: exactly 0
   -> 0, the pages only name > 0 and < 0).  ||r|| is kept as fp16 (reading: the
   pages do not list it, but the unbiased estimator needs it; fp16 like n).
3. Estimator ([juejin §2]; [freelamp QJL]; [csdn QJL-3]): for a full-precision
   query q,
       est(q, x) = n16 * <Pi q, c[idx]> + rnorm16 * sqrt(pi/2) / m * <S q, sigma>,
   sigma_j = 2 bit_j - 1.  The first term equals <q, x_hat>.  The constant is
   not printed on the pages; it is the unique one that makes the correction
   unbiased: for s ~ N(0, I_d), E[sign(<s, r>) <s, q>] = sqrt(2/pi) <r, q> / ||r||,
   so E_S[rnorm * sqrt(pi/2)/m * <S q, sign(S r)>] = <q, r> and E[est] = <q, x>.
4. Attention over compressed keys ([juejin §3]): logit = scale * est; softmax
   over the cached positions; output = sum_i p_i v_hat_i, where v_hat is the
   MSE-only reconstruction n_v16 * Pi_v^T c_v[idx_v] or the plain bf16 value.
   Query head h reads KV head h // (Hq / Hkv) (reading: contiguous GQA groups).
5. Search ([juejin §3]; [juejin §4]): est for every (query, vector) pair, sorted
   by score descending, equal scores by index ascending, first k kept.

The packed layout is the library's public contract (the header of the C-ABI):
bit (j mod 32) of word j // 32 of plane p holds bit p of idx_j; bit (j mod 32)
of sign word j // 32 holds bit_j; pad bits are 0.
"""

from __future__ import annotations

from dataclasses import dataclass
from math import pi, sqrt
from typing import Optional

import numpy as np

from .codebook import Codebook

QJL_CONST = sqrt(pi / 2.0)


def fp16_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest IEEE binary16 value (ties to even), returned as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


@dataclass
class Quantized:
    """Codes of n vectors: idx [n, d] (int), norm16 [n], and for the QJL stage
    signs [n, m] (bool) and rnorm16 [n]."""

    idx: np.ndarray
    norm16: np.ndarray
    signs: Optional[np.ndarray] = None
    rnorm16: Optional[np.ndarray] = None


def scalar_codes(U: np.ndarray, cb: Codebook) -> np.ndarray:
    """Index of the nearest centroid = number of thresholds strictly below u."""
    return np.searchsorted(cb.thresholds, U, side="left").astype(np.int64)


def dequantize(idx: np.ndarray, norm16: np.ndarray, Pi: np.ndarray, cb: Codebook) -> np.ndarray:
    """x_hat = n16 * Pi^T c[idx] (row form: (c[idx] @ Pi) scaled by n16)."""
    return norm16[..., None] * (cb.centroids[idx] @ Pi)


def qjl_signs(X: np.ndarray, idx: np.ndarray, norm16: np.ndarray, Pi: np.ndarray,
              S: np.ndarray, cb: Codebook) -> tuple[np.ndarray, np.ndarray]:
    """Residual r = x - x_hat, its fp16 norm and the sign bits of S r (step 2)."""
    R = np.asarray(X, dtype=np.float64) - dequantize(idx, norm16, Pi, cb)
    rnorm16 = fp16_round(np.linalg.norm(R, axis=-1))
    signs = (R @ S.T) > 0.0
    return signs, rnorm16


def quantize(X: np.ndarray, Pi: np.ndarray, cb: Codebook, S: Optional[np.ndarray] = None) -> Quantized:
    """Steps 1 and 2 for the rows of X (any float dtype, computed in float64).

    ``S`` None means the MSE-only mode (no QJL stage).
    """
    X = np.asarray(X, dtype=np.float64)
    n = np.linalg.norm(X, axis=-1)
    norm16 = fp16_round(n)
    Y = X @ Pi.T
    safe = np.where(n > 0, n, 1.0)
    U = np.where((n > 0)[..., None], Y / safe[..., None], 0.0)
    idx = scalar_codes(U, cb)
    if S is None:
        return Quantized(idx=idx, norm16=norm16)
    signs, rnorm16 = qjl_signs(X, idx, norm16, Pi, S, cb)
    return Quantized(idx=idx, norm16=norm16, signs=signs, rnorm16=rnorm16)


# ----------------------------------------------------------------------------- packing

def _words(nbits: int) -> int:
    return (nbits + 31) // 32


def pack_bits(B: np.ndarray) -> np.ndarray:
    """[..., nbits] bools -> [..., ceil(nbits/32)] uint32, bit j%32 of word j//32."""
    B = np.asarray(B, dtype=bool)
    nb = B.shape[-1]
    W = _words(nb)
    pad = np.zeros(B.shape[:-1] + (W * 32,), dtype=np.uint64)
    pad[..., :nb] = B
    pad = pad.reshape(B.shape[:-1] + (W, 32))
    weights = (np.uint64(1) << np.arange(32, dtype=np.uint64))
    return (pad * weights).sum(axis=-1).astype(np.uint32)


def unpack_bits(words: np.ndarray, nbits: int) -> np.ndarray:
    words = np.asarray(words, dtype=np.uint32)
    j = np.arange(nbits)
    return ((words[..., j // 32] >> (j % 32).astype(np.uint32)) & 1).astype(bool)


def pack_planes(idx: np.ndarray, bits: int) -> np.ndarray:
    """idx [..., d] -> planes uint32 [..., bits, W]: plane p holds bit p of each idx_j."""
    idx = np.asarray(idx, dtype=np.int64)
    return np.stack([pack_bits((idx >> p) & 1) for p in range(bits)], axis=-2)


def unpack_planes(planes: np.ndarray, d: int) -> np.ndarray:
    planes = np.asarray(planes, dtype=np.uint32)
    bits = planes.shape[-2]
    idx = np.zeros(planes.shape[:-2] + (d,), dtype=np.int64)
    for p in range(bits):
        idx |= unpack_bits(planes[..., p, :], d).astype(np.int64) << p
    return idx


def pack_signs(signs: np.ndarray) -> np.ndarray:
    return pack_bits(signs)


def unpack_signs(words: np.ndarray, m: int) -> np.ndarray:
    return unpack_bits(words, m)


# ----------------------------------------------------------------------------- estimator

def estimate(q: np.ndarray, z: Quantized, Pi: np.ndarray, cb: Codebook,
             S: Optional[np.ndarray] = None) -> np.ndarray:
    """est(q, x) for one query q [d] against every coded vector in z (step 3)."""
    q = np.asarray(q, dtype=np.float64)
    mse = z.norm16 * (cb.centroids[z.idx] @ (Pi @ q))
    if S is None:
        return mse
    m = S.shape[0]
    sigma = 2.0 * z.signs.astype(np.float64) - 1.0
    return mse + z.rnorm16 * (QJL_CONST / m) * (sigma @ (S @ q))


def estimate_all(Q: np.ndarray, z: Quantized, Pi: np.ndarray, cb: Codebook,
                 S: Optional[np.ndarray] = None) -> np.ndarray:
    """est for every (query row of Q, coded vector) pair -> [nq, n]."""
    return np.stack([estimate(q, z, Pi, cb, S) for q in np.asarray(Q, dtype=np.float64)])


def _group(h: int, Hq: int, Hkv: int) -> int:
    return h // (Hq // Hkv)


def attention_logits(q: np.ndarray, keys: Quantized, lens: np.ndarray, Pi: np.ndarray,
                     S: np.ndarray, cb: Codebook, scale: float) -> np.ndarray:
    """logits [B, Hq, N]: scale * est(q[b, h], key[b, h // G, i]) for i < lens[b], NaN beyond.

    keys carries idx [B, Hkv, N, d], norm16 [B, Hkv, N], signs [B, Hkv, N, m], rnorm16 [B, Hkv, N];
    S None (and no signs) means MSE-only keys, est = n16 <Pi q, c[idx]>.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, _ = q.shape
    Hkv, N = keys.idx.shape[1], keys.idx.shape[2]
    out = np.full((B, Hq, N), np.nan)
    for b in range(B):
        L = int(lens[b])
        for h in range(Hq):
            g = _group(h, Hq, Hkv)
            z = Quantized(idx=keys.idx[b, g, :L], norm16=keys.norm16[b, g, :L])
            if S is not None:
                z.signs, z.rnorm16 = keys.signs[b, g, :L], keys.rnorm16[b, g, :L]
            out[b, h, :L] = scale * estimate(q[b, h], z, Pi, cb, S)
    return out


def softmax(logits: np.ndarray) -> np.ndarray:
    """Softmax of a 1-D array with the maximum subtracted first."""
    e = np.exp(logits - np.max(logits))
    return e / np.sum(e)


def attention_values(logits: np.ndarray, lens: np.ndarray, Hkv: int,
                     values_dense: Optional[np.ndarray] = None, values: Optional[Quantized] = None,
                     Pi_v: Optional[np.ndarray] = None, cb_v: Optional[Codebook] = None) -> np.ndarray:
    """o [B, Hq, d] = sum_{i < lens[b]} softmax(logits[b, h, :lens[b]])_i v_hat_i; zeros when lens[b] == 0.

    Values are either dense [B, Hkv, N, d] (``values_dense``) or MSE-only codes
    (``values`` with idx and norm16, rotation ``Pi_v`` and table ``cb_v``).
    """
    B, Hq, _ = logits.shape
    d = values_dense.shape[-1] if values_dense is not None else Pi_v.shape[0]
    out = np.zeros((B, Hq, d))
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        for h in range(Hq):
            g = _group(h, Hq, Hkv)
            p = softmax(np.asarray(logits[b, h, :L], dtype=np.float64))
            if values_dense is not None:
                V = np.asarray(values_dense[b, g, :L], dtype=np.float64)
            else:
                V = dequantize(values.idx[b, g, :L], values.norm16[b, g, :L], Pi_v, cb_v)
            out[b, h] = p @ V
    return out


def attention_output(q: np.ndarray, keys: Quantized, lens: np.ndarray, Pi: np.ndarray,
                     S: np.ndarray, cb: Codebook, scale: float,
                     values_dense: Optional[np.ndarray] = None,
                     values: Optional[Quantized] = None, Pi_v: Optional[np.ndarray] = None,
                     cb_v: Optional[Codebook] = None) -> np.ndarray:
    """Logits over the compressed keys, then the softmax-weighted value sum (attention_values)."""
    logits = attention_logits(q, keys, lens, Pi, S, cb, scale)
    return attention_values(logits, lens, keys.idx.shape[1], values_dense, values, Pi_v, cb_v)


# ----------------------------------------------------------------------------- search

def search_topk(Q: np.ndarray, db: Quantized, Pi: np.ndarray, cb: Codebook,
                S: Optional[np.ndarray], k: int) -> tuple[np.ndarray, np.ndarray]:
    """Top-k of est over the database for each query: scores [nq, k], indices [nq, k].

    Order: score descending, then index ascending (stable sort of the negated scores).
    """
    n = db.idx.shape[0]
    k = min(k, n)
    scores = estimate_all(Q, db, Pi, cb, S)
    top_s = np.empty((scores.shape[0], k))
    top_i = np.empty((scores.shape[0], k), dtype=np.int64)
    for r in range(scores.shape[0]):
        order = np.argsort(-scores[r], kind="stable")[:k]
        top_s[r] = scores[r, order]
        top_i[r] = order
    return top_s, top_i


def recall_at_1(top_idx: np.ndarray, true_top1: np.ndarray) -> float:
    """Recall@1@k: fraction of queries whose true nearest neighbour is among the k returned."""
    top_idx = np.asarray(top_idx)
    hits = [(true_top1[r] in top_idx[r]) for r in range(top_idx.shape[0])]
    return float(np.mean(hits))


# ----------------------------------------------------------------------------- fractional bit widths

@dataclass
class SplitCodebook:
    """Fractional bit width ([juejin §4]: KV quality at 3.5 and 2.5 bits per channel).

    Reading (the pages give only the per-channel averages): the first ``d_hi``
    rotated coordinates are coded with the (b+1)-bit table ``hi``, the other
    d - d_hi with the b-bit table ``lo``; both are the Lloyd-Max tables of the
    same one-coordinate law, which is exact because the rotated coordinates are
    exchangeable.  Average MSE bits b + d_hi / d; the QJL stage adds 1 bit.
    """

    lo: Codebook
    hi: Codebook
    d_hi: int

    def hi_mask(self, d: int) -> np.ndarray:
        return np.arange(d) < self.d_hi

    def codes(self, U: np.ndarray) -> np.ndarray:
        """Per coordinate: the number of its table's thresholds strictly below u."""
        hi = self.hi_mask(U.shape[-1])
        return np.where(hi, scalar_codes(U, self.hi), scalar_codes(U, self.lo))

    def centroid_values(self, idx: np.ndarray) -> np.ndarray:
        """c_{g(j)}[idx_j] for every coordinate j."""
        hi = self.hi_mask(idx.shape[-1])
        return np.where(hi, self.hi.centroids[np.minimum(idx, len(self.hi.centroids) - 1)],
                        self.lo.centroids[np.minimum(idx, len(self.lo.centroids) - 1)])


def split_quantize(X: np.ndarray, Pi: np.ndarray, scb: SplitCodebook, S: Optional[np.ndarray] = None) -> Quantized:
    """Steps 1 and 2 with the split table: as ``quantize`` coordinate by coordinate."""
    X = np.asarray(X, dtype=np.float64)
    n = np.linalg.norm(X, axis=-1)
    norm16 = fp16_round(n)
    Y = X @ Pi.T
    safe = np.where(n > 0, n, 1.0)
    U = np.where((n > 0)[..., None], Y / safe[..., None], 0.0)
    idx = scb.codes(U)
    if S is None:
        return Quantized(idx=idx, norm16=norm16)
    R = X - split_dequantize(idx, norm16, Pi, scb)
    rnorm16 = fp16_round(np.linalg.norm(R, axis=-1))
    return Quantized(idx=idx, norm16=norm16, signs=(R @ S.T) > 0.0, rnorm16=rnorm16)


def split_dequantize(idx: np.ndarray, norm16: np.ndarray, Pi: np.ndarray, scb: SplitCodebook) -> np.ndarray:
    """x_hat = n16 * Pi^T c_g[idx]."""
    return norm16[..., None] * (scb.centroid_values(idx) @ Pi)


def split_estimate(q: np.ndarray, z: Quantized, Pi: np.ndarray, scb: SplitCodebook,
                   S: Optional[np.ndarray] = None) -> np.ndarray:
    """The estimator of step 3 with the split table."""
    q = np.asarray(q, dtype=np.float64)
    mse = z.norm16 * (scb.centroid_values(z.idx) @ (Pi @ q))
    if S is None:
        return mse
    m = S.shape[0]
    sigma = 2.0 * z.signs.astype(np.float64) - 1.0
    return mse + z.rnorm16 * (QJL_CONST / m) * (sigma @ (S @ q))


def pack_split(idx: np.ndarray, b: int, d_hi: int) -> np.ndarray:
    """Packed row of a split code (the library's layout): the b planes of all d coordinates
    ([..., b * W] words, plane p = bit p of idx_j), then plane b of the first d_hi
    coordinates ([..., ceil(d_hi / 32)] words)."""
    idx = np.asarray(idx, dtype=np.int64)
    low = pack_planes(idx & ((1 << b) - 1), b)
    low = low.reshape(low.shape[:-2] + (-1,))
    top = pack_bits(((idx[..., :d_hi] >> b) & 1).astype(bool))
    return np.concatenate([low, top], axis=-1)


def unpack_split(words: np.ndarray, d: int, b: int, d_hi: int) -> np.ndarray:
    words = np.asarray(words, dtype=np.uint32)
    W = _words(d)
    low = words[..., :b * W].reshape(words.shape[:-1] + (b, W))
    idx = unpack_planes(low, d)
    top = unpack_bits(words[..., b * W:], d_hi).astype(np.int64)
    idx[..., :d_hi] |= top << b
    return idx
