"""Shared helpers of the GPU parity tests: contexts built from oracle matrices, the parity
rules, and conversions between the packed device layout and the oracle's arrays."""
from math import sqrt

import numpy as np
import torch

import oracle
from oracle.codebook import sphere_codebook

# Parity rules (floating point):  logits and outputs within relative 1e-3 or absolute 1e-4;
# a code may differ only where the oracle's u lies within 1e-5 of a threshold; a sign only
# where |(S r)_j| < 1e-5 * n; stored fp16 norms within one fp16 ulp.
REL, ABS = 1e-3, 1e-4
CODE_BAND = 1e-5


class Pair:
    """A libtq context and the oracle pieces that use the same float32 matrices."""

    def __init__(self, d, bits, mode=0, seed=0, m=None):
        from compressed_kv_cache_02_b300 import tq
        self.d = d
        P = bits - 1 if mode == tq.TQ_MODE_PROD else bits
        m = d if m is None else m
        Pi, S = oracle.method_matrices(seed, d, m if mode == tq.TQ_MODE_PROD else 1)
        self.Pi32 = Pi.astype(np.float32)
        self.S32 = S.astype(np.float32) if mode == tq.TQ_MODE_PROD else None
        self.ctx = tq.Context(d, bits, seed=seed, mode=mode, m=m, Pi=self.Pi32, S=self.S32)
        self.Pi = self.Pi32.astype(np.float64)
        self.S = None if self.S32 is None else self.S32.astype(np.float64)
        self.cb = sphere_codebook(d, P)
        self.P = P
        self.m = m if mode == tq.TQ_MODE_PROD else 0

    # oracle side
    def oquant(self, X):
        return oracle.quantize(np.asarray(X, dtype=np.float64), self.Pi, self.cb, self.S)

    def to_device(self, z, lead_shape):
        """Oracle codes -> packed device Codes with leading shape lead_shape."""
        from compressed_kv_cache_02_b300 import tq
        planes = oracle.pack_planes(z.idx, self.P).view(np.int32)
        norm = z.norm16.astype(np.float16).view(np.int16)
        codes = tq.Codes(planes=torch.from_numpy(planes.reshape(*lead_shape, self.P, -1).copy()).cuda(),
                         norm=torch.from_numpy(norm.reshape(lead_shape).copy()).cuda())
        if self.S is not None:
            codes.signs = torch.from_numpy(oracle.pack_signs(z.signs).view(np.int32).reshape(*lead_shape, -1).copy()).cuda()
            codes.rnorm = torch.from_numpy(z.rnorm16.astype(np.float16).view(np.int16).reshape(lead_shape).copy()).cuda()
        return codes

    def from_device(self, codes):
        """Packed device Codes -> (idx, norm16, signs, rnorm16) numpy, rows flattened."""
        planes = codes.planes.cpu().numpy().view(np.uint32)
        planes = planes.reshape(-1, self.P, planes.shape[-1])
        idx = oracle.unpack_planes(planes, self.d)
        n16 = codes.norm.cpu().numpy().view(np.float16).reshape(-1).astype(np.float64)
        if codes.signs is None:
            return idx, n16, None, None
        signs = oracle.unpack_signs(codes.signs.cpu().numpy().view(np.uint32).reshape(idx.shape[0], -1), self.m)
        r16 = codes.rnorm.cpu().numpy().view(np.float16).reshape(-1).astype(np.float64)
        return idx, n16, signs, r16


def fp16_ulps(a, b):
    ia = np.asarray(a, dtype=np.float64).astype(np.float16).view(np.int16).astype(np.int64)
    ib = np.asarray(b, dtype=np.float64).astype(np.float16).view(np.int16).astype(np.int64)
    return np.abs(ia - ib)


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    ok = (err <= ABS) | (err <= REL * np.abs(ref))
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside rel {REL}/abs {ABS}; "
                             f"first {bad.tolist()}: got {got[tuple(bad[0])]}, ref {ref[tuple(bad[0])]}")


def check_codes(pair, X, codes):
    """Quantize parity of device codes against the oracle on the same rows X [n, d].
    Returns the boolean mask of rows whose encodings are identical."""
    X = np.asarray(X, dtype=np.float64).reshape(-1, pair.d)
    z = pair.oquant(X)
    idx, n16, signs, r16 = pair.from_device(codes)
    assert idx.shape == z.idx.shape
    n = np.linalg.norm(X, axis=1)
    U = np.where(n[:, None] > 0, (X @ pair.Pi.T) / np.where(n > 0, n, 1)[:, None], 0.0)
    near = np.min(np.abs(U[..., None] - pair.cb.thresholds[None, None, :]), axis=-1) < CODE_BAND
    diff = idx != z.idx
    assert not (diff & ~near).any(), f"{int((diff & ~near).sum())} codes differ away from a threshold"
    assert fp16_ulps(n16, z.norm16).max(initial=0) <= 1
    same = ~diff.any(axis=1) & (n16 == z.norm16)
    if signs is not None:
        # signs of the GPU's own codes and norm: oracle residual built from them
        s_own, r_own = oracle.qjl_signs(X, idx, n16, pair.Pi, pair.S, pair.cb)
        R = X - oracle.dequantize(idx, n16, pair.Pi, pair.cb)
        z_own = R @ pair.S.T
        sd = signs != s_own
        assert not (sd & ~(np.abs(z_own) < CODE_BAND * n[:, None])).any(), "sign bits differ away from 0"
        assert fp16_ulps(r16, r_own).max(initial=0) <= 1
        same &= ~(signs != z.signs).any(axis=1) & (r16 == z.rnorm16)
    return same
