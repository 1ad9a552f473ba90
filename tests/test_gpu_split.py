"""GPU parity of split (fractional bit width) contexts against the oracle: codes of tq_quantize
(CUDA-core kernel), logits of tq_attn_logits on oracle-coded keys, decode appends, and the calls
that refuse split contexts.  3.5 bits per channel = 2 MSE bits with the first half of the rotated
coordinates at 3, plus 1 QJL bit; 2.5 = 1 MSE bit with half at 2, plus 1 QJL bit."""
from math import sqrt

import numpy as np
import pytest
import torch

import oracle
from oracle.codebook import sphere_codebook
from compressed_kv_cache_02_b300 import inputs
from gpu_helpers import CODE_BAND, assert_close, fp16_ulps

pytestmark = pytest.mark.gpu


def _tq():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from compressed_kv_cache_02_b300 import tq
    return tq


class SplitPair:
    """A split libtq context and the oracle pieces on the same float32 matrices."""

    def __init__(self, d, bits, d_hi, mode=0, seed=0):
        tq = _tq()
        self.d, self.d_hi = d, d_hi
        self.P = bits - 1 if mode == tq.TQ_MODE_PROD else bits
        prod = mode == tq.TQ_MODE_PROD
        Pi, S = oracle.method_matrices(seed, d, d if prod else 1)
        self.Pi32 = Pi.astype(np.float32)
        self.S32 = S.astype(np.float32) if prod else None
        self.ctx = tq.Context(d, bits, seed=seed, mode=mode, m=d, Pi=self.Pi32, S=self.S32, d_hi=d_hi)
        self.Pi = self.Pi32.astype(np.float64)
        self.S = None if self.S32 is None else self.S32.astype(np.float64)
        self.m = d if prod else 0
        self.scb = oracle.SplitCodebook(lo=sphere_codebook(d, self.P), hi=sphere_codebook(d, self.P + 1), d_hi=d_hi)

    def oquant(self, X):
        return oracle.split_quantize(np.asarray(X, dtype=np.float64), self.Pi, self.scb, self.S)

    def to_device(self, z, lead):
        tq = _tq()
        words = oracle.pack_split(z.idx, self.P, self.d_hi).view(np.int32)
        codes = tq.Codes(planes=torch.from_numpy(words.reshape(*lead, -1).copy()).cuda(),
                         norm=torch.from_numpy(z.norm16.astype(np.float16).view(np.int16).reshape(lead).copy()).cuda())
        if self.S is not None:
            codes.signs = torch.from_numpy(oracle.pack_signs(z.signs).view(np.int32).reshape(*lead, -1).copy()).cuda()
            codes.rnorm = torch.from_numpy(z.rnorm16.astype(np.float16).view(np.int16).reshape(lead).copy()).cuda()
        return codes

    def check_codes(self, X, codes):
        """Device codes of rows X against the oracle (the parity rules of gpu_helpers)."""
        X = np.asarray(X, dtype=np.float64).reshape(-1, self.d)
        z = self.oquant(X)
        words = codes.planes.cpu().numpy().view(np.uint32).reshape(X.shape[0], -1)
        assert words.shape[1] == self.ctx.row_words
        idx = oracle.unpack_split(words, self.d, self.P, self.d_hi)
        n16 = codes.norm.cpu().numpy().view(np.float16).reshape(-1).astype(np.float64)
        n = np.linalg.norm(X, axis=1)
        U = np.where(n[:, None] > 0, (X @ self.Pi.T) / np.where(n > 0, n, 1)[:, None], 0.0)
        hi = np.arange(self.d) < self.d_hi
        dist_hi = np.min(np.abs(U[..., None] - self.scb.hi.thresholds[None, None, :]), axis=-1)
        dist_lo = np.min(np.abs(U[..., None] - self.scb.lo.thresholds[None, None, :]), axis=-1)
        near = np.where(hi, dist_hi, dist_lo) < CODE_BAND
        diff = idx != z.idx
        assert not (diff & ~near).any(), f"{int((diff & ~near).sum())} codes differ away from a threshold"
        assert fp16_ulps(n16, z.norm16).max(initial=0) <= 1
        same = ~diff.any(axis=1) & (n16 == z.norm16)
        if self.S is not None:
            signs = oracle.unpack_signs(codes.signs.cpu().numpy().view(np.uint32).reshape(X.shape[0], -1), self.m)
            r16 = codes.rnorm.cpu().numpy().view(np.float16).reshape(-1).astype(np.float64)
            R = X - oracle.split_dequantize(idx, n16, self.Pi, self.scb)   # the GPU's own reconstruction
            zr = R @ self.S.T
            assert not ((signs != (zr > 0)) & ~(np.abs(zr) < CODE_BAND * n[:, None])).any(), "signs differ away from 0"
            assert fp16_ulps(r16, np.linalg.norm(R, axis=1)).max(initial=0) <= 1
            same &= ~(signs != z.signs).any(axis=1) & (r16 == z.rnorm16)
        return same


CASES = [  # d, bits, d_hi, mode
    (128, 3, 64, 0),    # 3.5 bits per channel (2.5 MSE + 1 QJL)
    (128, 2, 64, 0),    # 2.5 bits per channel (1.5 MSE + 1 QJL)
    (128, 4, 32, 0),    # 3 MSE bits with a quarter at 4
    (200, 3, 96, 0),    # d = 200 (7 words, top plane of 3 words)
    (128, 2, 96, 1),    # MSE-only: 2 bits with three quarters at 3
]


@pytest.mark.parametrize("d,bits,d_hi,mode", CASES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_split_quantize(d, bits, d_hi, mode, dtype):
    pr = SplitPair(d, bits, d_hi, mode, seed=2)
    n = 1037
    X = inputs.gaussian(n, d, seed=21)
    if dtype == "bf16":
        X = X.to(torch.bfloat16)
    codes = pr.ctx.quantize(X.cuda())
    assert pr.ctx.sync_status() == 0
    same = pr.check_codes(X.float().numpy(), codes)
    assert same.mean() > 0.97


@pytest.mark.parametrize("bits,d_hi,mode", [(3, 64, 0), (2, 64, 0), (4, 32, 0), (2, 96, 1)])
@pytest.mark.parametrize("path", ["cuda_core", "tensor"])
def test_split_quantize_bulk_bf16(bits, d_hi, mode, path):
    """Bulk bf16 rows at d = 128: the tcgen05 quantize kernel (AUTO/TENSOR) and the CUDA-core one."""
    tq = _tq()
    pr = SplitPair(128, bits, d_hi, mode, seed=12)
    pr.ctx.set_kernel_path(tq.TQ_PATH_TENSOR if path == "tensor" else tq.TQ_PATH_CUDA_CORE)
    fac = inputs.anisotropic_factors(1, 128, seed=13)
    X = inputs.anisotropic(1, 1, 5003, 128, fac, seed=13)[0, 0]
    codes = pr.ctx.quantize(X.cuda())
    assert pr.ctx.sync_status() == 0
    same = pr.check_codes(X.float().numpy(), codes)
    assert same.mean() > 0.97


@pytest.mark.parametrize("d,bits,d_hi,mode", CASES)
def test_split_logits(d, bits, d_hi, mode):
    pr = SplitPair(d, bits, d_hi, mode, seed=3)
    B, Hkv, G, N, lens = 2, 2, 4, 1100, [1100, 517]
    fac = inputs.anisotropic_factors(Hkv, d, seed=4)
    K = inputs.anisotropic(B, Hkv, N, d, fac, seed=4)
    Q = inputs.anisotropic(B, Hkv, G, d, fac, seed=5, dtype=torch.float32).reshape(B, Hkv * G, d)
    z = pr.oquant(K.float().numpy().reshape(-1, d))
    keys = pr.to_device(z, (B, Hkv, N))
    scale = 1.0 / sqrt(d)
    length = torch.tensor(lens, dtype=torch.int32).cuda()
    got = pr.ctx.attn_logits(Q.cuda(), keys, N, length, scale).cpu().numpy()
    assert pr.ctx.sync_status() == 0
    idx = z.idx.reshape(B, Hkv, N, d)
    for b in range(B):
        for h in range(Hkv * G):
            kvh = h // G
            sl = slice((b * Hkv + kvh) * N, (b * Hkv + kvh) * N + lens[b])
            zz = oracle.Quantized(idx=idx[b, kvh, :lens[b]], norm16=z.norm16[sl],
                                  signs=None if z.signs is None else z.signs[sl],
                                  rnorm16=None if z.rnorm16 is None else z.rnorm16[sl])
            ref = scale * oracle.split_estimate(Q[b, h].numpy(), zz, pr.Pi, pr.scb, pr.S)
            assert_close(got[b, h, :lens[b]], ref, "split logits")


def test_split_append_writes_the_row_at_len():
    tq = _tq()
    pr = SplitPair(128, 3, 64, 0, seed=6)
    B, H, cap = 3, 2, 40
    cache = pr.ctx.alloc_codes(B, H, cap)
    lens = torch.tensor([0, 7, 39], dtype=torch.int32).cuda()
    x = inputs.gaussian(B * H, 128, seed=7).reshape(B, H, 128).cuda()
    pr.ctx.append(x, cache, cap, lens)
    assert pr.ctx.sync_status() == 0
    for b, L in enumerate([0, 7, 39]):
        for h in range(H):
            codes = tq.Codes(planes=cache.planes[b, h, L:L + 1], norm=cache.norm[b, h, L:L + 1],
                             signs=cache.signs[b, h, L:L + 1], rnorm=cache.rnorm[b, h, L:L + 1])
            pr.check_codes(x[b, h].cpu().numpy()[None], codes)
    # every other row is untouched (zero)
    mask = torch.ones(B, H, cap, dtype=torch.bool, device="cuda")
    for b, L in enumerate([0, 7, 39]):
        mask[b, :, L] = False
    assert int(cache.planes[mask].abs().sum()) == 0


def test_split_contexts_are_refused_where_unsupported():
    tq = _tq()
    pr = SplitPair(128, 3, 64, 0, seed=8)
    db = pr.ctx.quantize(inputs.gaussian(64, 128, seed=9).cuda())
    with pytest.raises(tq.TQError) as e:
        pr.ctx.search_topk(inputs.gaussian(2, 128, seed=10).cuda(), db, 4)
    assert e.value.code == tq.TQ_ERR_UNSUPPORTED
    keys = pr.ctx.alloc_codes(1, 1, 64)
    q = torch.zeros(1, 4, 128, device="cuda")
    length = torch.tensor([64], dtype=torch.int32, device="cuda")
    with pytest.raises(tq.TQError) as e:
        pr.ctx.attn_output(q, keys, 64, length, 1.0, torch.zeros(1, 1, 64, 128, dtype=torch.bfloat16, device="cuda"))
    assert e.value.code == tq.TQ_ERR_UNSUPPORTED


@pytest.mark.parametrize("vbits,d_hi,lens", [(3, 64, [1500, 333]), (2, 64, [1500, 1]), (1, 96, [700, 1500]),
                                            (2, 32, [0, 1500])])
def test_split_values(vbits, d_hi, lens):
    """Softmax + value sum over split (fractional bit width) MSE value codes: 2.5 MSE bits per
    value channel = 2 bits with half the rotated coordinates at 3, and so on."""
    tq = _tq()
    d, B, Hkv, G, N = 128, 2, 2, 4, 1500
    pr = SplitPair(d, vbits, d_hi, mode=tq.TQ_MODE_MSE, seed=31)
    fac = inputs.anisotropic_factors(Hkv, d, seed=32)
    V = inputs.anisotropic(B, Hkv, N, d, fac, seed=32)
    z = pr.oquant(V.float().numpy().reshape(-1, d))
    vcodes = pr.to_device(z, (B, Hkv, N))
    g = np.random.default_rng(33)
    logits = g.normal(0, 2.0, size=(B, Hkv * G, N)).astype(np.float32)
    length = torch.tensor(lens, dtype=torch.int32).cuda()
    got = tq.attn_values(torch.from_numpy(logits).cuda(), length, vcodes, vctx=pr.ctx).cpu().numpy()
    assert pr.ctx.sync_status() == 0
    idx = z.idx.reshape(B, Hkv, N, d)
    n16 = z.norm16.reshape(B, Hkv, N)
    for b in range(B):
        for h in range(Hkv * G):
            L = lens[b]
            if L == 0:
                assert np.all(got[b, h] == 0)
                continue
            p = oracle.turboquant.softmax(logits[b, h, :L].astype(np.float64))
            Vh = oracle.split_dequantize(idx[b, h // G, :L], n16[b, h // G, :L], pr.Pi, pr.scb)
            assert_close(got[b, h], p @ Vh, "split values")
