"""GPU parity of the libtq kernels against the oracle, through the C-ABI.

Inputs come from the seeded generators; the oracle's codes are packed and fed to the
attention and search kernels so both sides score identical encodings, and separate
end-to-end checks compare rows whose encodings agree."""
from math import sqrt

import numpy as np
import pytest
import torch

import oracle
from compressed_kv_cache_02_b300 import inputs
from gpu_helpers import Pair, assert_close, check_codes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from compressed_kv_cache_02_b300 import tq  # noqa: F401  (fails loudly without libtq.so)


def _tq():
    from compressed_kv_cache_02_b300 import tq
    return tq


# ------------------------------------------------------------------ quantization

@pytest.mark.parametrize("d,bits,n", [(128, 3, 4096), (128, 4, 777), (200, 2, 1000), (200, 4, 513),
                                      (33, 3, 300), (300, 3, 100), (8, 2, 65)])
def test_quantize_fp32_gaussian(d, bits, n):
    pr = Pair(d, bits)
    X = inputs.gaussian(n, d, seed=0).cuda()
    codes = pr.ctx.quantize(X)
    assert pr.ctx.sync_status() == 0
    same = check_codes(pr, X.cpu().numpy(), codes)
    assert same.mean() > 0.99


@pytest.mark.parametrize("bits", [3, 4, 5])
def test_quantize_bf16_anisotropic(bits):
    d = 128
    pr = Pair(d, bits, seed=4)
    fac = inputs.anisotropic_factors(2, d, seed=4)
    X = inputs.anisotropic(1, 2, 1500, d, fac, seed=4)
    codes = pr.ctx.quantize(X.cuda())
    same = check_codes(pr, X.float().numpy().reshape(-1, d), codes)
    assert same.mean() > 0.99


@pytest.mark.parametrize("mode,bits", [(0, 2), (0, 3), (0, 4), (0, 5), (1, 1), (1, 2), (1, 3), (1, 4)])
@pytest.mark.parametrize("n,ld", [(4096, 128), (5003, 128), (4500, 136), (4200, 128)])
def test_quantize_bulk_bf16(mode, bits, n, ld, kernel_path):
    """Bulk bf16 rows at d=128: tcgen05 tensor-core path (n >= 4096) and CUDA-core path."""
    tq = _tq()
    pr = Pair(128, bits, mode=mode, seed=12)
    pr.ctx.set_kernel_path(tq.TQ_PATH_TENSOR if kernel_path == "tensor" else tq.TQ_PATH_CUDA_CORE)
    fac = inputs.anisotropic_factors(1, ld, seed=12)
    X = inputs.anisotropic(1, 1, n, ld, fac, seed=13)[0, 0]          # rows of ld values; the first 128 are used
    X[7] = 0.0                                                        # zero rows: one inside, the last
    X[n - 1] = 0.0
    Xd = X.cuda()[:, :128]
    codes = pr.ctx.quantize(Xd)
    assert pr.ctx.sync_status() == 0
    same = check_codes(pr, X[:, :128].float().numpy(), codes)
    assert same.mean() > 0.99
    idx, n16, signs, r16 = pr.from_device(codes)
    for r in (7, n - 1):
        assert n16[r] == 0
        if mode == 0:
            assert r16[r] == 0 and not signs[r].any()


def test_quantize_bulk_norm_overflow_flag():
    """The tensor-core quantizer flags a norm that rounds to fp16 infinity, and the rest stays coded."""
    tq = _tq()
    pr = Pair(128, 3, seed=12)
    pr.ctx.set_kernel_path(tq.TQ_PATH_TENSOR)
    X = inputs.gaussian(4200, 128, seed=14).to(torch.bfloat16)
    X[4100] = 1.0e4                                                   # ||x|| = 1.1e5 > fp16 max
    codes = pr.ctx.quantize(X.cuda())
    assert pr.ctx.sync_status() == tq.TQ_DEVERR_NORM_OVERFLOW
    keep = np.ones(4200, dtype=bool)
    keep[4100] = False
    idx, n16, signs, r16 = pr.from_device(codes)
    assert np.isinf(n16[4100])
    rows = torch.from_numpy(np.nonzero(keep)[0]).cuda()
    sub = tq.Codes(codes.planes[rows], codes.norm[rows], codes.signs[rows], codes.rnorm[rows])
    same = check_codes(pr, X.float().numpy()[keep], sub)
    assert same.mean() > 0.99


@pytest.mark.parametrize("bits,d,n", [(1, 128, 700), (3, 128, 700), (4, 128, 700), (5, 128, 700), (6, 200, 300),
                                      (8, 128, 700), (8, 128, 5000), (7, 33, 250), (8, 300, 90)])
def test_quantize_mse_mode(bits, d, n):
    """MSE-mode codes at every width 1..8 (5..8 bits: the table read from device memory), the
    decode-append (small n) and bulk (n >= 4736) variants of the CUDA-core kernel."""
    tq = _tq()
    pr = Pair(d, bits, mode=tq.TQ_MODE_MSE, seed=1)
    X = inputs.gaussian(n, d, seed=5).cuda()
    codes = pr.ctx.quantize(X)
    assert codes.signs is None
    assert pr.ctx.sync_status() == 0
    same = check_codes(pr, X.cpu().numpy(), codes)
    assert same.mean() > 0.9


@pytest.mark.parametrize("d", [128, 200])
def test_round_trip_at_eight_bits_on_gpu(d):
    """The high-bit-width round trip through the library: the codes of x at 8 MSE bits, the
    reconstruction of those codes (oracle), coded again by the library.  The second coding passes
    the quantize parity rules against the oracle's coding of the same reconstruction, and returns
    the first codes on every row whose centroid vector has unit norm to within 5e-3 (the rows
    where the renormalisation of re-coding keeps every value in its cell; over 99 % of them)."""
    tq = _tq()
    pr = Pair(d, 8, mode=tq.TQ_MODE_MSE, seed=3)
    X = 5.0 * inputs.gaussian(1000, d, seed=11)
    c1 = pr.ctx.quantize(X.cuda())
    idx1, n1, _, _ = pr.from_device(c1)
    Xh = oracle.dequantize(idx1, n1, pr.Pi, pr.cb).astype(np.float32)
    c2 = pr.ctx.quantize(torch.from_numpy(Xh).cuda())
    assert pr.ctx.sync_status() == 0
    check_codes(pr, Xh, c2)
    idx2, _, _, _ = pr.from_device(c2)
    unit = np.abs(np.linalg.norm(pr.cb.centroids[idx1], axis=1) - 1.0) < 5e-3
    assert unit.mean() > 0.99
    assert np.array_equal(idx2[unit], idx1[unit])
    Xd = X.numpy().astype(np.float64)
    rel = np.sum((Xd - Xh) ** 2, axis=1) / np.sum(Xd ** 2, axis=1)
    assert abs(rel.mean() - pr.cb.distortion()) < 3 * rel.std() / np.sqrt(len(rel)) + 2.0 ** -22


def test_quantize_strided_rows_zero_rows_and_empty():
    pr = Pair(64, 3)
    X = inputs.gaussian(40, 96, seed=6)
    X[3] = 0.0
    Xc = X.cuda()
    sub = Xc[:, 10:74]                     # row stride 96 > d
    codes = pr.ctx.quantize(sub)
    check_codes(pr, X[:, 10:74].numpy(), codes)
    idx, n16, signs, r16 = pr.from_device(codes)
    assert n16[3] == 0 and r16[3] == 0 and not signs[3].any()
    empty = pr.ctx.alloc_codes(0)
    pr.ctx.quantize(Xc[:0, :64], out=empty)
    assert pr.ctx.sync_status() == 0


def test_norm_overflow_sets_device_flag():
    tq = _tq()
    pr = Pair(16, 3)
    X = torch.full((2, 16), 1.0e5).cuda()   # ||x|| = 4e5 > fp16 max
    pr.ctx.quantize(X)
    assert pr.ctx.sync_status() == tq.TQ_DEVERR_NORM_OVERFLOW
    assert pr.ctx.sync_status() == 0        # cleared by the previous read


def test_argument_errors_raise():
    tq = _tq()
    pr = Pair(16, 3)
    X = inputs.gaussian(4, 16, seed=1).cuda()
    with pytest.raises(TypeError):
        pr.ctx.quantize(X.double())
    out = pr.ctx.alloc_codes(4)
    code = tq.lib.tq_quantize(pr.ctx.h, X.data_ptr(), 0, 4, 8, out.planes.data_ptr(), out.signs.data_ptr(),
                              out.norm.data_ptr(), out.rnorm.data_ptr(), None)
    assert code == tq.TQ_ERR_ARG                                   # ld_x < d
    code = tq.lib.tq_quantize(pr.ctx.h, X.data_ptr(), 0, 4, 16, out.planes.data_ptr(), None,
                              out.norm.data_ptr(), None, None)
    assert code == tq.TQ_ERR_ARG                                   # PROD needs signs
    with pytest.raises(tq.TQError):
        tq.Context(16, 6)                                          # PROD mode: at most 4 MSE bits
    with pytest.raises(tq.TQError):
        tq.Context(16, 9, mode=tq.TQ_MODE_MSE)                     # MSE mode: at most 8 bits


# ------------------------------------------------------------------ attention

def _kv_case(B, Hkv, G, N, d, kbits, vmode, seed, lens, vbits=3):
    """Oracle-coded keys (and values) on the device plus the oracle's reference pieces."""
    tq = _tq()
    kp = Pair(d, kbits, seed=seed)
    fac = inputs.anisotropic_factors(Hkv, d, seed=seed)
    K = inputs.anisotropic(B, Hkv, N, d, fac, seed=seed)
    V = inputs.anisotropic(B, Hkv, N, d, inputs.anisotropic_factors(Hkv, d, seed=seed + 1000), seed=seed + 1000)
    Q = inputs.anisotropic(B, Hkv, G, d, fac, seed=seed + 2000, dtype=torch.float32)
    q = Q.reshape(B, Hkv * G, d)
    kz = kp.oquant(K.float().numpy())
    keys = kp.to_device(kz, (B, Hkv, N))
    case = dict(kp=kp, K=K, V=V, q=q, kz=kz, keys=keys, lens=np.array(lens), B=B, Hkv=Hkv, Hq=Hkv * G, N=N, d=d)
    if vmode == "mse":
        vp = Pair(d, vbits, mode=tq.TQ_MODE_MSE, seed=seed + 7)
        vz = vp.oquant(V.float().numpy())
        case.update(vp=vp, vz=vz, vcodes=vp.to_device(vz, (B, Hkv, N)))
    return case


def _run_logits(c, scale):
    length = torch.tensor(c["lens"], dtype=torch.int32).cuda()
    return c["kp"].ctx.attn_logits(c["q"].cuda(), c["keys"], c["N"], length, scale)


@pytest.fixture(params=["cuda_core", "tensor"])
def kernel_path(request):
    return request.param


@pytest.mark.parametrize("B,Hkv,G,N,d,bits,lens", [
    (1, 1, 16, 4096, 128, 3, [4096]),            # tiny correctness workload: 16 queries x 4096 keys
    (1, 8, 4, 1100, 128, 4, [1100]),             # decode layer shape (4-bit keys), ragged tail
    (2, 2, 4, 1500, 128, 3, [1500, 731]),        # long-context shape (3-bit keys), two lengths
    (1, 2, 6, 300, 128, 3, [300]),               # GQA group of 6: a padded head quad
    (2, 1, 4, 400, 200, 2, [400, 0]),            # d=200 (7 words), an empty sequence
    (1, 2, 4, 257, 300, 3, [257]),               # d=300: generic (table-free) path
    (1, 1, 4, 100, 33, 5, [100]),                # ragged d, 4 MSE bits
    (1, 2, 4, 999, 100, 2, [999]),               # d=100 on the d<=128 path, 1 MSE bit
    (1, 1, 4, 2049, 128, 5, [2049]),             # 4 MSE bits on the d<=128 path
    # capacities that are multiples of 8: the bulk-copy tensor-core path takes these
    (2, 2, 4, 1504, 128, 3, [1500, 731]),        # ragged lengths inside 32-key units
    (1, 8, 4, 1104, 128, 4, [1100]),             # 3 MSE bits
    (1, 2, 6, 304, 128, 3, [300]),               # padded head quad
    (1, 2, 4, 1000, 100, 2, [999]),              # d=100, 1 MSE bit
    (3, 2, 4, 4104, 128, 3, [4100, 33, 0]),      # long, short and empty sequences in one launch
])
def test_logits(B, Hkv, G, N, d, bits, lens, kernel_path):
    tq = _tq()
    c = _kv_case(B, Hkv, G, N, d, bits, None, seed=3, lens=lens)
    c["kp"].ctx.set_kernel_path(tq.TQ_PATH_TENSOR if kernel_path == "tensor" else tq.TQ_PATH_CUDA_CORE)
    scale = 1.0 / sqrt(d)
    got = _run_logits(c, scale).cpu().numpy()
    assert c["kp"].ctx.sync_status() == 0
    ref = oracle.attention_logits(c["q"].numpy(), c["kz"], c["lens"], c["kp"].Pi, c["kp"].S, c["kp"].cb, scale)
    for b in range(B):
        L = lens[b]
        assert_close(got[b, :, :L], ref[b, :, :L], "logits")


@pytest.mark.parametrize("bits", [3, 6, 8])
def test_logits_mse_keys(kernel_path, bits):
    tq = _tq()
    d, N = 128, 600
    kp = Pair(d, bits, mode=tq.TQ_MODE_MSE, seed=9)
    kp.ctx.set_kernel_path(tq.TQ_PATH_TENSOR if kernel_path == "tensor" else tq.TQ_PATH_CUDA_CORE)
    K = inputs.gaussian(2 * N, d, seed=9).reshape(1, 2, N, d)
    q = inputs.gaussian(8, d, seed=10).reshape(1, 8, d)
    kz = kp.oquant(K.numpy())
    keys = kp.to_device(kz, (1, 2, N))
    got = kp.ctx.attn_logits(q.cuda(), keys, N, torch.tensor([N], dtype=torch.int32).cuda(), 0.5).cpu().numpy()
    ref = oracle.attention_logits(q.numpy(), kz, np.array([N]), kp.Pi, None, kp.cb, 0.5)
    assert_close(got, ref, "mse-key logits")


@pytest.mark.parametrize("vmode", ["bf16", "mse", "mse8"])
@pytest.mark.parametrize("B,Hkv,G,N,bits,lens", [
    (1, 8, 4, 1100, 4, [1100]),
    (2, 2, 4, 2600, 3, [2600, 1]),
    (2, 1, 6, 700, 3, [0, 699]),
])
def test_attention_output(vmode, B, Hkv, G, N, bits, lens):
    d = 128
    c = _kv_case(B, Hkv, G, N, d, bits, "mse" if vmode == "mse8" else vmode, seed=11, lens=lens,
                 vbits=8 if vmode == "mse8" else 3)
    scale = 1.0 / sqrt(d)
    length = torch.tensor(lens, dtype=torch.int32).cuda()
    kp = c["kp"]
    if vmode == "bf16":
        got = kp.ctx.attn_output(c["q"].cuda(), c["keys"], N, length, scale, c["V"].cuda())
        ref = oracle.attention_output(c["q"].numpy(), c["kz"], c["lens"], kp.Pi, kp.S, kp.cb, scale,
                                      values_dense=c["V"].float().numpy())
    else:
        vp = c["vp"]
        got = kp.ctx.attn_output(c["q"].cuda(), c["keys"], N, length, scale, c["vcodes"], vctx=vp.ctx)
        ref = oracle.attention_output(c["q"].numpy(), c["kz"], c["lens"], kp.Pi, kp.S, kp.cb, scale,
                                      values=c["vz"], Pi_v=vp.Pi, cb_v=vp.cb)
    assert kp.ctx.sync_status() == 0
    assert_close(got.cpu().numpy(), ref, "attention output")


@pytest.mark.parametrize("vmode", ["bf16", "mse"])
@pytest.mark.parametrize("B,Hkv,G,N,lens", [(1, 8, 4, 1100, [1100]), (2, 2, 4, 2600, [2600, 1]),
                                           (2, 1, 6, 700, [0, 699])])
def test_attention_values_from_logits(vmode, B, Hkv, G, N, lens):
    """The softmax + value step on its own: oracle logits in, weighted values out."""
    tq = _tq()
    d = 128
    c = _kv_case(B, Hkv, G, N, d, 3, vmode, seed=13, lens=lens)
    kp = c["kp"]
    ref_l = oracle.attention_logits(c["q"].numpy(), c["kz"], c["lens"], kp.Pi, kp.S, kp.cb, 1.0 / sqrt(d))
    logits = torch.from_numpy(np.nan_to_num(ref_l, nan=0.0).astype(np.float32)).cuda()
    length = torch.tensor(lens, dtype=torch.int32).cuda()
    if vmode == "bf16":
        got = tq.attn_values(logits, length, c["V"].cuda())
        ref = oracle.attention_values(logits.cpu().numpy(), c["lens"], Hkv, values_dense=c["V"].float().numpy())
    else:
        vp = c["vp"]
        got = tq.attn_values(logits, length, c["vcodes"], vctx=vp.ctx)
        ref = oracle.attention_values(logits.cpu().numpy(), c["lens"], Hkv, values=c["vz"], Pi_v=vp.Pi, cb_v=vp.cb)
    torch.cuda.synchronize()
    assert_close(got.cpu().numpy(), ref, "softmax-weighted values")


@pytest.mark.parametrize("vbits,d", [(1, 128), (2, 128), (3, 112), (4, 128), (4, 100), (5, 128), (8, 128), (8, 100),
                                     (6, 200)])
def test_attention_values_code_widths(vbits, d):
    """The value sum at every MSE width: 1-4 bits on the d <= 128 coded-value kernel, 5-8 bits (and
    d = 200) on the generic one with the table from device memory; head dims below 128 (padded
    coordinates)."""
    tq = _tq()
    B, Hkv, G, N, lens = 2, 2, 4, 1500, [1500, 333]
    c = _kv_case(B, Hkv, G, N, d, 3, "mse", seed=17, lens=lens, vbits=vbits)
    kp, vp = c["kp"], c["vp"]
    ref_l = oracle.attention_logits(c["q"].numpy(), c["kz"], c["lens"], kp.Pi, kp.S, kp.cb, 1.0 / sqrt(d))
    logits = torch.from_numpy(np.nan_to_num(ref_l, nan=0.0).astype(np.float32)).cuda()
    length = torch.tensor(lens, dtype=torch.int32).cuda()
    got = tq.attn_values(logits, length, c["vcodes"], vctx=vp.ctx)
    ref = oracle.attention_values(logits.cpu().numpy(), c["lens"], Hkv, values=c["vz"], Pi_v=vp.Pi, cb_v=vp.cb)
    torch.cuda.synchronize()
    assert_close(got.cpu().numpy(), ref, f"values at {vbits} bits, d = {d}")


@pytest.mark.parametrize("vbits,d,B,Hkv,G,N,lens", [
    (3, 128, 2, 2, 4, 1500, [1500, 333]),       # several chunks, a ragged tail
    (3, 128, 3, 1, 6, 700, [700, 1, 0]),       # a padded head quad, a 1-key and an empty sequence
    (2, 128, 1, 2, 4, 5000, [4999]),
    (1, 112, 1, 2, 4, 2100, [2100]),
    (3, 100, 2, 1, 4, 900, [900, 31]),
])
def test_attention_values_tensor_cores(vbits, d, B, Hkv, G, N, lens):
    """The tcgen05 value sum (TQ_PATH_TENSOR on the value context): bit masks transposed per
    block of 32 keys, Walsh terms as e4m3 A in tensor memory, the softmax weights as e4m3 pieces,
    two-pass softmax per chunk; against the oracle."""
    tq = _tq()
    c = _kv_case(B, Hkv, G, N, d, 3, "mse", seed=37, lens=lens, vbits=vbits)
    kp, vp = c["kp"], c["vp"]
    vp.ctx.set_kernel_path(tq.TQ_PATH_TENSOR)
    ref_l = oracle.attention_logits(c["q"].numpy(), c["kz"], c["lens"], kp.Pi, kp.S, kp.cb, 1.0 / sqrt(d))
    logits = torch.from_numpy(np.nan_to_num(ref_l, nan=0.0).astype(np.float32)).cuda()
    length = torch.tensor(lens, dtype=torch.int32).cuda()
    got = tq.attn_values(logits, length, c["vcodes"], vctx=vp.ctx)
    assert vp.ctx.sync_status() == 0
    ref = oracle.attention_values(logits.cpu().numpy(), c["lens"], Hkv, values=c["vz"], Pi_v=vp.Pi, cb_v=vp.cb)
    assert_close(got.cpu().numpy(), ref, f"tensor-core values at {vbits} bits, d = {d}")
    # the partial states of the same path merge to the same output
    part = tq.attn_values_partial(logits, length, c["vcodes"], vctx=vp.ctx)
    merged = tq.attn_merge_partials(part[None], vctx=vp.ctx)
    torch.cuda.synchronize()
    assert_close(merged.cpu().numpy(), ref, "tensor-core values through the partial states")


def test_decode_append_and_advance():
    """Decode-step append: every appended row lands at position len[b] + s of its (batch, head)
    and passes the quantize parity rules there (codes by the threshold band, signs on the GPU's
    own codes, norm and residual norm within one fp16 ulp); every other slot keeps the zeros of
    the freshly allocated cache."""
    tq = _tq()
    d, B, H, cap = 128, 2, 3, 40
    L0 = [5, 17]
    pr = Pair(d, 3, seed=2)
    cache = pr.ctx.alloc_codes(B, H, cap)
    length = torch.tensor(L0, dtype=torch.int32).cuda()
    steps = [inputs.gaussian(B * H, d, seed=100 + s).reshape(B, H, d) for s in range(3)]
    for x in steps:
        pr.ctx.append(x.cuda(), cache, cap, length)
        pr.ctx.advance_len(length, cap)
    assert pr.ctx.sync_status() == 0
    assert length.cpu().tolist() == [L + len(steps) for L in L0]
    written = torch.zeros(B, H, cap, dtype=torch.bool)
    for s, x in enumerate(steps):
        pos = [L + s for L in L0]
        rows = tq.Codes(planes=torch.stack([cache.planes[b, :, pos[b]] for b in range(B)]).reshape(B * H, pr.P, -1),
                        norm=torch.stack([cache.norm[b, :, pos[b]] for b in range(B)]).reshape(B * H),
                        signs=torch.stack([cache.signs[b, :, pos[b]] for b in range(B)]).reshape(B * H, -1),
                        rnorm=torch.stack([cache.rnorm[b, :, pos[b]] for b in range(B)]).reshape(B * H))
        check_codes(pr, x.numpy().reshape(B * H, d), rows)
        for b in range(B):
            written[b, :, pos[b]] = True
    for field in (cache.planes, cache.signs, cache.norm, cache.rnorm):
        f = field.cpu()
        assert not f[~written].any(), "a slot other than len[b] + step was written"
    # an out-of-range length is flagged and skipped, not written
    bad = torch.tensor([cap, 0], dtype=torch.int32).cuda()
    before = cache.planes.clone()
    pr.ctx.append(steps[0].cuda(), cache, cap, bad)
    assert pr.ctx.sync_status() == tq.TQ_DEVERR_LEN_RANGE
    assert torch.equal(cache.planes[0], before[0])
    pr.ctx.advance_len(torch.tensor([cap], dtype=torch.int32).cuda(), cap)
    assert pr.ctx.sync_status() == tq.TQ_DEVERR_LEN_RANGE


def test_end_to_end_quantize_then_logits():
    d, N, G = 128, 2048, 4
    pr = Pair(d, 3, seed=21)
    K = inputs.gaussian(N, d, seed=21).reshape(1, 1, N, d)
    q = inputs.gaussian(G, d, seed=22).reshape(1, G, d)
    codes = pr.ctx.quantize(K.cuda().reshape(N, d))
    same = check_codes(pr, K.numpy().reshape(N, d), codes)
    keys = _tq().Codes(planes=codes.planes.reshape(1, 1, N, pr.P, -1), norm=codes.norm.reshape(1, 1, N),
                       signs=codes.signs.reshape(1, 1, N, -1), rnorm=codes.rnorm.reshape(1, 1, N))
    got = pr.ctx.attn_logits(q.cuda(), keys, N, torch.tensor([N], dtype=torch.int32).cuda(), 1.0).cpu().numpy()
    kz = pr.oquant(K.numpy())
    ref = oracle.attention_logits(q.numpy(), kz, np.array([N]), pr.Pi, pr.S, pr.cb, 1.0)
    assert_close(got[0][:, same], ref[0][:, same], "end-to-end logits (rows with identical codes)")


# ------------------------------------------------------------------ search

def _topk_ok(got_s, got_i, ref_s, ref_i, all_scores):
    """Identical top-k sets apart from near-ties at the k-th score."""
    for r in range(ref_i.shape[0]):
        g, o = set(got_i[r].tolist()), set(ref_i[r].tolist())
        kth = ref_s[r, -1]
        tol = max(1e-4, 1e-3 * abs(kth))
        for i in g ^ o:
            assert abs(all_scores[r, i] - kth) <= tol, f"query {r}: item {i} differs away from a tie"
        assert np.all(np.diff(got_s[r]) <= 0)
        assert_close(got_s[r], all_scores[r, got_i[r]], "returned scores")


@pytest.mark.parametrize("d,bits,n,nq,k", [(200, 2, 5000, 13, 10), (200, 4, 3000, 8, 100), (128, 3, 4096, 16, 1),
                                         (200, 4, 1000, 5, 128), (64, 2, 300, 3, 50),
                                         # several 16-query groups and row chunks, ragged last tile and group
                                         (200, 2, 20011, 40, 100), (128, 3, 9001, 33, 7), (256, 4, 6000, 17, 64),
                                         (200, 3, 130, 20, 128)])
def test_search_topk(d, bits, n, nq, k, kernel_path):
    tq = _tq()
    pr = Pair(d, bits, seed=5)
    pr.ctx.set_kernel_path(tq.TQ_PATH_TENSOR if kernel_path == "tensor" else tq.TQ_PATH_CUDA_CORE)
    X = inputs.cone(n, d, seed=5, mu_seed=77)
    Q = inputs.cone(nq, d, seed=6, mu_seed=77)
    z = pr.oquant(X.numpy())
    db = pr.to_device(z, (n,))
    s, i = pr.ctx.search_topk(Q.cuda(), db, k)
    assert pr.ctx.sync_status() == 0
    ref_s, ref_i = oracle.search_topk(Q.numpy(), z, pr.Pi, pr.cb, pr.S, k)
    scores = oracle.estimate_all(Q.numpy(), z, pr.Pi, pr.cb, pr.S)
    _topk_ok(s.cpu().numpy(), i.cpu().numpy().astype(np.int64), ref_s, ref_i, scores)


@pytest.mark.parametrize("bits,d,n,nq,k", [(2, 200, 3001, 21, 10), (3, 128, 2000, 17, 64), (1, 256, 1500, 5, 7)])
def test_search_topk_mse(bits, d, n, nq, k, kernel_path):
    """Search over MSE-mode codes of 1-3 bits (no QJL signs): the tcgen05 kernel with only its
    Walsh-term vectors (tensor path) and the byte-table kernel (CUDA-core path)."""
    tq = _tq()
    pr = Pair(d, bits, mode=tq.TQ_MODE_MSE, seed=6)
    pr.ctx.set_kernel_path(tq.TQ_PATH_TENSOR if kernel_path == "tensor" else tq.TQ_PATH_CUDA_CORE)
    X = inputs.cone(n, d, seed=15, mu_seed=77)
    Q = inputs.cone(nq, d, seed=16, mu_seed=77)
    z = pr.oquant(X.numpy())
    db = pr.to_device(z, (n,))
    s, i = pr.ctx.search_topk(Q.cuda(), db, k)
    assert pr.ctx.sync_status() == 0
    ref_s, ref_i = oracle.search_topk(Q.numpy(), z, pr.Pi, pr.cb, None, k)
    scores = oracle.estimate_all(Q.numpy(), z, pr.Pi, pr.cb, None)
    _topk_ok(s.cpu().numpy(), i.cpu().numpy().astype(np.int64), ref_s, ref_i, scores)


@pytest.mark.parametrize("bits,d", [(8, 200), (6, 64)])
def test_search_topk_wide_mse(bits, d):
    """Search over MSE-mode codes of 6 and 8 bits (generic scorer, table from device memory)."""
    tq = _tq()
    n, nq, k = 2000, 6, 20
    pr = Pair(d, bits, mode=tq.TQ_MODE_MSE, seed=5)
    X = inputs.cone(n, d, seed=5, mu_seed=77)
    Q = inputs.cone(nq, d, seed=6, mu_seed=77)
    z = pr.oquant(X.numpy())
    db = pr.to_device(z, (n,))
    s, i = pr.ctx.search_topk(Q.cuda(), db, k)
    assert pr.ctx.sync_status() == 0
    ref_s, ref_i = oracle.search_topk(Q.numpy(), z, pr.Pi, pr.cb, None, k)
    scores = oracle.estimate_all(Q.numpy(), z, pr.Pi, pr.cb, None)
    _topk_ok(s.cpu().numpy(), i.cpu().numpy().astype(np.int64), ref_s, ref_i, scores)


@pytest.mark.parametrize("d", [64, 128])
def test_search_ties_resolve_to_lower_index(d, kernel_path):
    tq = _tq()
    n = 600
    pr = Pair(d, 3, seed=8)
    pr.ctx.set_kernel_path(tq.TQ_PATH_TENSOR if kernel_path == "tensor" else tq.TQ_PATH_CUDA_CORE)
    X = inputs.cone(n, d, seed=8, mu_seed=1)
    X[400] = X[17]
    X[555] = X[17]
    z = pr.oquant(X.numpy())
    db = pr.to_device(z, (n,))
    Q = X[17:18].clone()
    s, i = pr.ctx.search_topk(Q.cuda(), db, 5)
    i = i.cpu().numpy()[0].tolist()
    s = s.cpu().numpy()[0]
    assert i.index(17) < i.index(400) < i.index(555)
    assert s[i.index(17)] == s[i.index(400)] == s[i.index(555)]
