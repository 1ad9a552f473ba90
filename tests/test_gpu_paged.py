"""GPU parity of the fused paged decode step (tq_paged_decode_step) against the oracle: the
appended rows against the oracle's codes of the new tokens (parity rules of gpu_helpers), the
output against the oracle's attention over the GPU's own pages (so a code that differs at a
threshold cannot move the comparison), untouched slots, and the advanced lengths; over several
consecutive steps, ragged lengths, a page boundary, the last slot of the table, and bf16 inputs
with two head quads per KV head."""
from math import sqrt

import numpy as np
import pytest
import torch

import oracle
from oracle import paged
from compressed_kv_cache_02_b300 import inputs
from gpu_helpers import Pair, assert_close, check_codes

pytestmark = pytest.mark.gpu
D = 128


def _tq():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from compressed_kv_cache_02_b300 import tq
    return tq


def _pools_from_device(cache, kp, vp):
    """GPU pools -> oracle pools (Quantized with [num_pages, Hkv, page_size, ...])."""
    NP, H, PS = cache.knorm.shape
    n = NP * H * PS
    kq = oracle.Quantized(
        idx=oracle.unpack_planes(cache.kplanes.cpu().numpy().view(np.uint32).reshape(n, kp.P, -1), D).reshape(NP, H, PS, D),
        norm16=cache.knorm.cpu().numpy().view(np.float16).astype(np.float64),
        signs=oracle.unpack_signs(cache.ksigns.cpu().numpy().view(np.uint32).reshape(n, -1), D).reshape(NP, H, PS, D),
        rnorm16=cache.krnorm.cpu().numpy().view(np.float16).astype(np.float64))
    vq = oracle.Quantized(
        idx=oracle.unpack_planes(cache.vplanes.cpu().numpy().view(np.uint32).reshape(n, vp.P, -1), D).reshape(NP, H, PS, D),
        norm16=cache.vnorm.cpu().numpy().view(np.float16).astype(np.float64))
    return kq, vq


def _prefill(cache, kp, vp, table, lens, ps, K, V):
    """Oracle codes of tokens 0 .. lens[b] - 1 written into their pages on the device."""
    kz = kp.oquant(K.reshape(-1, D))
    vz = vp.oquant(V.reshape(-1, D))
    B, H, N = K.shape[:3]
    kpl = oracle.pack_planes(kz.idx, kp.P).view(np.int32).reshape(B, H, N, kp.P, -1)
    ksg = oracle.pack_signs(kz.signs).view(np.int32).reshape(B, H, N, -1)
    kn = kz.norm16.astype(np.float16).view(np.int16).reshape(B, H, N)
    kr = kz.rnorm16.astype(np.float16).view(np.int16).reshape(B, H, N)
    vpl = oracle.pack_planes(vz.idx, vp.P).view(np.int32).reshape(B, H, N, vp.P, -1)
    vn = vz.norm16.astype(np.float16).view(np.int16).reshape(B, H, N)
    host = {k: getattr(cache, k).cpu().numpy() for k in ("kplanes", "ksigns", "knorm", "krnorm", "vplanes", "vnorm")}
    for b in range(B):
        for i in range(lens[b]):
            pg, sl = table[b][i // ps], i % ps
            host["kplanes"][pg, :, sl] = kpl[b, :, i]
            host["ksigns"][pg, :, sl] = ksg[b, :, i]
            host["knorm"][pg, :, sl] = kn[b, :, i]
            host["krnorm"][pg, :, sl] = kr[b, :, i]
            host["vplanes"][pg, :, sl] = vpl[b, :, i]
            host["vnorm"][pg, :, sl] = vn[b, :, i]
    for k, v in host.items():
        getattr(cache, k).copy_(torch.from_numpy(v))


@pytest.mark.parametrize("kbits,vbits,G,dtype", [(3, 3, 4, "f32"), (4, 2, 8, "bf16"), (2, 4, 4, "f32"), (3, 3, 6, "f32")])
def test_paged_decode_steps(kbits, vbits, G, dtype):
    tq = _tq()
    B, Hkv, ps, num_pages, max_pages, steps = 3, 2, 64, 24, 6, 3
    kp = Pair(D, kbits, seed=0)
    vp = Pair(D, vbits, mode=tq.TQ_MODE_MSE, seed=1)
    lens0 = np.array([0, 127, 381])          # empty, one before a page boundary, near the table's end
    rng = np.random.default_rng(kbits * 10 + vbits)
    pages = rng.permutation(num_pages)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    used = 0
    for b in range(B):
        need = (lens0[b] + steps + ps - 1) // ps
        table[b, :need] = pages[used:used + need]
        used += need
    N = int(lens0.max()) + steps
    fk = inputs.anisotropic_factors(Hkv, D, seed=3)
    fv = inputs.anisotropic_factors(Hkv, D, seed=4)
    K = inputs.anisotropic(B, Hkv, N, D, fk, seed=3).float().numpy()
    V = inputs.anisotropic(B, Hkv, N, D, fv, seed=4).float().numpy()
    cache = tq.alloc_paged_cache(kp.ctx, vp.ctx, num_pages, Hkv, ps)
    _prefill(cache, kp, vp, table, lens0, ps, K, V)
    tbl = torch.from_numpy(table).cuda()
    length = torch.from_numpy(lens0.astype(np.int32)).cuda()
    scale = 1.0 / sqrt(D)
    lens = lens0.copy()
    for s in range(steps):
        q = inputs.anisotropic(B, Hkv, G, D, fk, seed=100 + s, dtype=torch.float32).reshape(B, Hkv * G, D)
        kn = np.stack([K[b, :, lens[b]] for b in range(B)])
        vn = np.stack([V[b, :, lens[b]] for b in range(B)])
        tdt = torch.float32 if dtype == "f32" else torch.bfloat16
        kn_t, vn_t = torch.from_numpy(kn).to(tdt), torch.from_numpy(vn).to(tdt)
        out = tq.paged_decode_step(kp.ctx, vp.ctx, q.cuda(), kn_t.cuda(), vn_t.cuda(), cache, tbl, length, scale)
        assert kp.ctx.sync_status() == 0
        assert np.array_equal(length.cpu().numpy(), lens + 1)
        kq, vq = _pools_from_device(cache, kp, vp)
        # the appended rows: codes of the (rounded) new tokens
        for b in range(B):
            pg, sl = table[b][lens[b] // ps], lens[b] % ps
            rows = np.arange(Hkv)
            codes = tq.Codes(planes=cache.kplanes[pg, :, sl], norm=cache.knorm[pg, :, sl],
                             signs=cache.ksigns[pg, :, sl], rnorm=cache.krnorm[pg, :, sl])
            check_codes(kp, kn_t[b].float().numpy()[rows], codes)
            vcodes = tq.Codes(planes=cache.vplanes[pg, :, sl], norm=cache.vnorm[pg, :, sl])
            check_codes(vp, vn_t[b].float().numpy()[rows], vcodes)
        lens = lens + 1
        keys = paged.gather(kq, table, lens, ps)
        vals = paged.gather(vq, table, lens, ps)
        ref = oracle.attention_output(q.numpy(), keys, lens, kp.Pi, kp.S, kp.cb, scale, values=vals, Pi_v=vp.Pi, cb_v=vp.cb)
        assert_close(out.cpu().numpy(), ref, f"paged step {s}")
    # slots never written stay zero
    mask = np.ones((num_pages, Hkv, ps), dtype=bool)
    for b in range(B):
        for i in range(lens[b]):
            mask[table[b][i // ps], :, i % ps] = False
    assert int(np.abs(cache.kplanes.cpu().numpy()[mask]).sum()) == 0


def test_paged_step_flags_a_missing_page():
    tq = _tq()
    kp = Pair(D, 3, seed=0)
    vp = Pair(D, 3, mode=tq.TQ_MODE_MSE, seed=1)
    cache = tq.alloc_paged_cache(kp.ctx, vp.ctx, 4, 1, 32)
    tbl = torch.tensor([[0, -1]], dtype=torch.int32).cuda()     # position 32 has no page
    length = torch.tensor([32], dtype=torch.int32).cuda()
    q = torch.randn(1, 4, D).cuda()
    x = torch.randn(1, 1, D).cuda()
    tq.paged_decode_step(kp.ctx, vp.ctx, q, x, x, cache, tbl, length, 1.0)
    flags = kp.ctx.sync_status()
    assert flags & tq.TQ_DEVERR_LEN_RANGE
    assert int(length[0]) == 32   # no append, no advance


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """A wait that nothing completes (the self-test kernel) ends with TQ_DEVERR_TIMEOUT instead
    of hanging; the same context then quantizes normally."""
    tq = _tq()
    kp = Pair(D, 3, seed=0)
    assert tq.lib.tq_selftest_wait_timeout(kp.ctx.h, None) == tq.TQ_OK
    assert kp.ctx.sync_status() & tq.TQ_DEVERR_TIMEOUT
    x = torch.randn(8, D).cuda()
    codes = kp.ctx.quantize(x)
    assert kp.ctx.sync_status() == 0
    check_codes(kp, x.cpu().numpy(), codes)
