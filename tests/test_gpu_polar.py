"""GPU parity of the polar-angle encoder against the oracle: codes of tq_polar_quantize (an angle
code may differ only where the oracle's angle lies within the parity band of a threshold, scaled
by |x| over the radius it was taken at), stored radii and residual norms within one fp16 ulp,
signs of the GPU's own residual, scores of tq_polar_scores on oracle-coded keys within the
floating-point tolerance, and the two calls chained."""
from math import pi, sqrt

import numpy as np
import pytest
import torch

import oracle
from compressed_kv_cache_02_b300 import inputs
from gpu_helpers import CODE_BAND, assert_close, fp16_ulps

pytestmark = pytest.mark.gpu


def _tq():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from compressed_kv_cache_02_b300 import tq
    return tq


class PolarPair:
    def __init__(self, d, bits, qjl=True, seed=0):
        tq = _tq()
        Pi, S = oracle.method_matrices(seed, d, d)
        self.Pi32, self.S32 = Pi.astype(np.float32), S.astype(np.float32)
        self.ctx = tq.PolarContext(d, bits, qjl=qjl, Pi=self.Pi32, S=self.S32 if qjl else None)
        self.Pi = self.Pi32.astype(np.float64)
        self.S = self.S32.astype(np.float64) if qjl else None
        self.d, self.bits, self.qjl = d, bits, qjl
        self.pcb = oracle.polar_codebook(d, bits)

    def to_device(self, z):
        tq = _tq()
        codes = torch.from_numpy(oracle.pack_polar(z.codes, self.bits).view(np.int32).copy()).cuda()
        r16 = torch.from_numpy(z.r16.astype(np.float16).view(np.int16).copy()).cuda()
        out = tq.PolarCodes(codes=codes, r16=r16)
        if self.qjl:
            out.signs = torch.from_numpy(oracle.pack_signs(z.signs).view(np.int32).copy()).cuda()
            out.rnorm = torch.from_numpy(z.rnorm16.astype(np.float16).view(np.int16).copy()).cuda()
        return out

    def from_device(self, pc):
        codes = oracle.unpack_polar(pc.codes.cpu().numpy().view(np.uint32), self.d, self.bits)
        r16 = pc.r16.cpu().numpy().view(np.float16).astype(np.float64)
        if not self.qjl:
            return codes, r16, None, None
        signs = oracle.unpack_signs(pc.signs.cpu().numpy().view(np.uint32), self.d)
        rn = pc.rnorm.cpu().numpy().view(np.float16).astype(np.float64)
        return codes, r16, signs, rn

    def check_codes(self, X, pc):
        X = np.asarray(X, dtype=np.float64)
        z = oracle.polar_quantize(X, self.Pi, self.pcb, self.S)
        codes, r16, signs, rn = self.from_device(pc)
        n = np.linalg.norm(X, axis=1)
        _, angles, radii = oracle.polar_forward(X @ self.Pi.T)
        near = []
        for lev, (cb, ang, rad) in enumerate(zip(self.pcb.levels, angles, radii), start=1):
            band = CODE_BAND * n[:, None] / np.maximum(rad, 1e-30)
            dist = np.min(np.abs(ang[..., None] - cb.thresholds[None, None, :]), axis=-1)
            if lev == 1:   # the cut at 0 = 2 pi
                dist = np.minimum(dist, np.minimum(ang, 2 * pi - ang))
            near.append(dist < band)
        near = np.concatenate(near, axis=1)
        diff = codes != z.codes
        assert not (diff & ~near).any(), f"{int((diff & ~near).sum())} angle codes differ away from a threshold"
        assert fp16_ulps(r16, z.r16).max(initial=0) <= 1
        same = ~diff.any(axis=1) & (r16 == z.r16)
        if self.qjl:
            R = X - oracle.polar_dequantize(codes, r16, self.Pi, self.pcb)   # the GPU's own reconstruction
            zr = R @ self.S.T
            assert not ((signs != (zr > 0)) & ~(np.abs(zr) < CODE_BAND * n[:, None])).any(), "signs differ away from 0"
            assert fp16_ulps(rn, np.linalg.norm(R, axis=1)).max(initial=0) <= 1
            same &= ~(signs != z.signs).any(axis=1)
        return same


@pytest.mark.parametrize("d,bits,qjl", [(128, 3, True), (128, 2, True), (128, 4, False), (64, 1, True),
                                        (256, 3, True), (16, 2, True)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_polar_quantize(d, bits, qjl, dtype):
    pr = PolarPair(d, bits, qjl, seed=4)
    fac = inputs.anisotropic_factors(1, d, seed=5)
    X = inputs.anisotropic(1, 1, 1037, d, fac, seed=5)[0, 0]
    X = X.float() if dtype == "f32" else X.to(torch.bfloat16)
    pc = pr.ctx.quantize(X.cuda())
    assert pr.ctx.sync_status() == 0
    same = pr.check_codes(X.float().numpy(), pc)
    assert same.mean() > 0.97


def test_polar_quantize_zero_rows_and_strides():
    tq = _tq()
    pr = PolarPair(128, 3, True, seed=6)
    X = inputs.gaussian(40, 256, seed=7).cuda()
    X[3] = 0.0
    view = X[:, :128]                       # row stride 256
    pc = pr.ctx.quantize(view)
    assert pr.ctx.sync_status() == 0
    pr.check_codes(view.cpu().numpy(), pc)
    assert int(pc.r16[3]) == 0 and int(pc.codes[3].abs().sum()) == 0


@pytest.mark.parametrize("bits,qjl", [(1, True), (2, True), (3, True), (4, True), (2, False), (4, False)])
@pytest.mark.parametrize("path", ["tensor", "auto"])
def test_polar_quantize_tcgen05(bits, qjl, path):
    """The tensor-core encoder (bf16 rows at d = 128): forced on 1037 rows (8 full tiles of 128
    and a ragged tail of 13) with a zero row and a row stride of 192, or taken by AUTO on 4100
    rows (past the 4096-row cut, a tail of 4); same parity rules as the CUDA-core encoder."""
    tq = _tq()
    pr = PolarPair(128, bits, qjl, seed=14 + bits)
    n = 1037 if path == "tensor" else 4100
    if path == "tensor":
        pr.ctx.set_kernel_path(tq.TQ_PATH_TENSOR)
    fac = inputs.anisotropic_factors(1, 192, seed=15)
    X = inputs.anisotropic(1, 1, n, 192, fac, seed=15)[0, 0].to(torch.bfloat16).cuda()
    X[5] = 0.0
    view = X[:, :128] if path == "tensor" else X[:, :128].contiguous()
    pc = pr.ctx.quantize(view)
    assert pr.ctx.sync_status() == 0
    same = pr.check_codes(view.float().cpu().numpy(), pc)
    assert same.mean() > 0.97
    assert int(pc.r16[5]) == 0 and int(pc.codes[5].abs().sum()) == 0
    if qjl:
        assert int(pc.rnorm[5]) == 0 and int(pc.signs[5].abs().sum()) == 0


def test_polar_kernel_path_argument():
    tq = _tq()
    pr = PolarPair(64, 2, True, seed=3)
    with pytest.raises(tq.TQError):
        pr.ctx.set_kernel_path(7)
    pr.ctx.set_kernel_path(tq.TQ_PATH_TENSOR)   # d = 64: the CUDA-core encoder still runs
    X = torch.randn(50, 64, device="cuda", dtype=torch.bfloat16)
    pc = pr.ctx.quantize(X)
    assert pr.ctx.sync_status() == 0
    pr.check_codes(X.float().cpu().numpy(), pc)


@pytest.mark.parametrize("d,bits,qjl,nq", [(128, 3, True, 4), (128, 2, True, 6), (64, 4, False, 3),
                                           (256, 3, True, 5), (32, 1, True, 8)])
def test_polar_scores(d, bits, qjl, nq):
    pr = PolarPair(d, bits, qjl, seed=8)
    fac = inputs.anisotropic_factors(1, d, seed=9)
    K = inputs.anisotropic(1, 1, 1100, d, fac, seed=9)[0, 0].float().numpy()
    Q = inputs.anisotropic(1, 1, nq, d, fac, seed=10, dtype=torch.float32)[0, 0].numpy()
    z = oracle.polar_quantize(K, pr.Pi, pr.pcb, pr.S)
    keys = pr.to_device(z)
    scale = 1.0 / sqrt(d)
    got = pr.ctx.scores(torch.from_numpy(Q).cuda(), keys, scale).cpu().numpy()
    assert pr.ctx.sync_status() == 0
    for i in range(nq):
        ref = scale * oracle.polar_estimate(Q[i], z, pr.Pi, pr.pcb, pr.S)
        assert_close(got[i], ref, f"polar scores, query {i}")


def test_polar_quantize_then_score():
    pr = PolarPair(128, 3, True, seed=11)
    fac = inputs.anisotropic_factors(1, 128, seed=12)
    K = inputs.anisotropic(1, 1, 3000, 128, fac, seed=12)[0, 0]
    Q = inputs.anisotropic(1, 1, 4, 128, fac, seed=13, dtype=torch.float32)[0, 0]
    pc = pr.ctx.quantize(K.cuda())
    got = pr.ctx.scores(Q.cuda(), pc, 1.0).cpu().numpy()
    assert pr.ctx.sync_status() == 0
    codes, r16, signs, rn = pr.from_device(pc)
    z = oracle.PolarQuantized(codes=codes, r16=r16, signs=signs, rnorm16=rn)
    for i in range(4):
        assert_close(got[i], oracle.polar_estimate(Q[i].numpy(), z, pr.Pi, pr.pcb, pr.S), "chained polar scores")


@pytest.mark.parametrize("bits", [3, 2])
def test_polar_full_size_sampled(bits):
    """The measured workload (8 x 8 KV heads x 32768 keys, d=128, bf16 anisotropic) in the bench's
    launch shapes: codes of 512 sampled rows against the oracle, and scores of one 4-query group
    at 512 sampled keys against the oracle estimate from the GPU's own codes."""
    pr = PolarPair(128, bits, True, seed=0)
    Bf, Hf, Nf = 8, 8, 32768
    n = Bf * Hf * Nf
    fac = inputs.anisotropic_factors(Hf, 128, seed=2, device="cuda")
    X = inputs.anisotropic(Bf, Hf, Nf, 128, fac, seed=2, device="cuda").reshape(n, 128)
    q = inputs.anisotropic(Bf, Hf, 4, 128, fac, seed=2002, device="cuda", dtype=torch.float32).reshape(-1, 128)[:4]
    pc = pr.ctx.quantize(X)
    out = pr.ctx.scores(q, pc, 1.0)
    assert pr.ctx.sync_status() == 0
    g = np.random.default_rng(bits)
    rows = np.sort(g.choice(n, size=512, replace=False))
    ridx = torch.from_numpy(rows).cuda()
    tq = _tq()
    sub = tq.PolarCodes(pc.codes[ridx].cpu(), pc.r16[ridx].cpu(), pc.signs[ridx].cpu(), pc.rnorm[ridx].cpu())
    same = pr.check_codes(X[ridx].float().cpu().numpy(), sub)
    assert same.mean() > 0.97
    codes, r16, signs, rn = pr.from_device(sub)
    z = oracle.PolarQuantized(codes=codes, r16=r16, signs=signs, rnorm16=rn)
    got = out[:, ridx].cpu().numpy()
    for i in range(4):
        assert_close(got[i], oracle.polar_estimate(q[i].cpu().numpy(), z, pr.Pi, pr.pcb, pr.S), "full-size polar scores")


def test_polar_empty_calls():
    """n = 0 rows to quantize and n = 0 keys (or no queries) to score: nothing launches, OK."""
    tq = _tq()
    pr = PolarPair(64, 2, True, seed=3)
    empty = torch.zeros(0, 64, device="cuda")
    pc = pr.ctx.quantize(empty)
    assert pc.codes.shape == (0, pr.ctx.code_words)
    out = pr.ctx.scores(torch.randn(4, 64, device="cuda"), pc, 1.0)
    assert out.shape == (4, 0)
    keys = pr.ctx.quantize(torch.randn(10, 64, device="cuda"))
    assert pr.ctx.scores(torch.zeros(0, 64, device="cuda"), keys, 1.0).shape == (0, 10)
    assert pr.ctx.sync_status() == 0
