"""Parity at full workload sizes, in the launch configuration the benchmark times, on
sampled outputs the oracle computes one by one.

* Long-context decode: batch 8 x 8 KV heads x 131072 cached keys (d=128), keys 2+1 bits,
  values 3-bit MSE, 32 query heads.  The whole cache is quantized and scored on the GPU; the
  oracle re-codes sampled key rows from the same seeded inputs, recomputes sampled logits,
  and recomputes the full attention output of two (batch, head) pairs.
* Vector search: 10^6 database vectors (d=200, cone law) at 2 and 4 bits, 10^4 queries, top-100;
  the oracle scores the whole database for a few sampled queries.
* One decode layer of an 8B-class GQA model: 8 KV heads x 32768 keys (d=128), keys 4 bits
  (3 MSE + 1 QJL) quantized on the GPU, bf16 values, 32 query heads; the fused output and the
  logits of sampled heads against the oracle.
"""
from math import sqrt

import numpy as np
import pytest
import torch

import oracle
from compressed_kv_cache_02_b300 import inputs
from gpu_helpers import Pair, assert_close, check_codes

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

B, HKV, G, D, N0 = 8, 8, 4, 128, 131072
HQ = HKV * G
SEED = 3


@pytest.fixture(scope="module")
def decode_state():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from compressed_kv_cache_02_b300 import tq
    kp = Pair(D, 3, seed=0)
    vp = Pair(D, 3, mode=tq.TQ_MODE_MSE, seed=1)
    cap = N0 + 4096
    kc = kp.ctx.alloc_codes(B, HKV, cap)
    vc = vp.ctx.alloc_codes(B, HKV, cap)
    kfac = inputs.anisotropic_factors(HKV, D, seed=SEED, device="cuda")
    vfac = inputs.anisotropic_factors(HKV, D, seed=SEED + 1000, device="cuda")
    for b in range(B):
        K = inputs.anisotropic(1, HKV, N0, D, kfac, seed=SEED * 100 + b, device="cuda")
        V = inputs.anisotropic(1, HKV, N0, D, vfac, seed=SEED * 100 + 1000 + b, device="cuda")
        for h in range(HKV):
            kp.ctx.quantize(K[0, h], out=tq.Codes(kc.planes[b, h, :N0], kc.norm[b, h, :N0], kc.signs[b, h, :N0],
                                                  kc.rnorm[b, h, :N0]))
            vp.ctx.quantize(V[0, h], out=tq.Codes(vc.planes[b, h, :N0], vc.norm[b, h, :N0]))
        del K, V
    q = inputs.anisotropic(B, HKV, G, D, kfac, seed=30_000, device="cuda", dtype=torch.float32).reshape(B, HQ, D)
    length = torch.full((B,), N0, dtype=torch.int32, device="cuda")
    scale = 1.0 / sqrt(D)
    logits = kp.ctx.attn_logits(q, kc, cap, length, scale)
    out = tq.attn_values(logits, length, vc, vctx=vp.ctx)
    torch.cuda.synchronize()
    assert kp.ctx.sync_status() == 0 and vp.ctx.sync_status() == 0
    return dict(tq=tq, kp=kp, vp=vp, kc=kc, vc=vc, cap=cap, kfac=kfac, vfac=vfac, q=q.cpu(), logits=logits,
                out=out.cpu().numpy(), scale=scale)


def _rows(tensor_bh, idx):
    return tensor_bh[idx].cpu()


def _raw(fac, b, h, seed_base):
    """The same seeded rows the cache was built from (one batch row), on the CPU."""
    X = inputs.anisotropic(1, HKV, N0, D, fac, seed=seed_base + b, device="cuda")
    return X[0, h].float().cpu().numpy()


def test_sampled_key_codes_and_logits(decode_state):
    s = decode_state
    tq, kp, kc = s["tq"], s["kp"], s["kc"]
    rng = np.random.default_rng(0)
    for b, kvh in [(0, 0), (5, 3), (7, 7)]:
        X = _raw(s["kfac"], b, kvh, SEED * 100)
        rows = np.sort(rng.choice(N0, size=512, replace=False))
        sel = torch.from_numpy(rows).cuda()
        codes = tq.Codes(planes=kc.planes[b, kvh][sel], norm=kc.norm[b, kvh][sel], signs=kc.signs[b, kvh][sel],
                         rnorm=kc.rnorm[b, kvh][sel])
        same = check_codes(kp, X[rows], codes)
        assert same.mean() > 0.99
        z = kp.oquant(X[rows])
        got = s["logits"][b, kvh * G:(kvh + 1) * G][:, sel].cpu().numpy()
        for g in range(G):
            ref = s["scale"] * oracle.estimate(s["q"][b, kvh * G + g].numpy(), z, kp.Pi, kp.cb, kp.S)
            assert_close(got[g][same], ref[same], "sampled full-size logits")


def test_full_attention_output_of_sampled_heads(decode_state):
    s = decode_state
    kp, vp = s["kp"], s["vp"]
    for b, h in [(2, 9), (6, 30)]:
        kvh = h // G
        K = _raw(s["kfac"], b, kvh, SEED * 100)
        V = _raw(s["vfac"], b, kvh, SEED * 100 + 1000)
        kz = kp.oquant(K)
        vz = vp.oquant(V)
        logit = s["scale"] * oracle.estimate(s["q"][b, h].numpy(), kz, kp.Pi, kp.cb, kp.S)
        p = oracle.turboquant.softmax(logit)
        ref = p @ oracle.dequantize(vz.idx, vz.norm16, vp.Pi, vp.cb)
        assert_close(s["out"][b, h], ref, "full-size attention output")


@pytest.mark.parametrize("bits", [2, 4])
def test_search_full_database_sampled_queries(bits):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    d, n, nq, k = 200, 1_000_000, 10_000, 100
    pr = Pair(d, bits, seed=0)
    X = inputs.cone(n, d, seed=5, mu_seed=55, device="cuda")
    Q = inputs.cone(nq, d, seed=6, mu_seed=55, device="cuda")
    db = pr.ctx.quantize(X)
    top_s, top_i = pr.ctx.search_topk(Q, db, k)
    torch.cuda.synchronize()
    assert pr.ctx.sync_status() == 0
    Xc = X.cpu().numpy()
    z = pr.oquant(Xc)              # the oracle's own codes of the whole database
    for r in (0, 4321, 9999):
        q = Q[r].cpu().numpy()
        scores = oracle.estimate(q, z, pr.Pi, pr.cb, pr.S)
        order = np.argsort(-scores, kind="stable")[:k]
        got = top_i[r].cpu().numpy().astype(np.int64)
        kth = scores[order[-1]]
        tol = max(1e-4, 1e-3 * abs(kth))
        for i in set(got.tolist()) ^ set(order.tolist()):
            assert abs(scores[i] - kth) <= tol, f"query {r}: item {i} differs away from a tie"


def test_decode_layer_32k_bf16_values():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from compressed_kv_cache_02_b300 import tq
    hkv, n, seed = 8, 32768, 2
    kp = Pair(D, 4, seed=0)
    kfac = inputs.anisotropic_factors(hkv, D, seed=seed, device="cuda")
    vfac = inputs.anisotropic_factors(hkv, D, seed=seed + 1000, device="cuda")
    K = inputs.anisotropic(1, hkv, n, D, kfac, seed=seed, device="cuda")
    V = inputs.anisotropic(1, hkv, n, D, vfac, seed=seed + 1000, device="cuda")
    q = inputs.anisotropic(1, hkv, G, D, kfac, seed=seed + 2000, device="cuda", dtype=torch.float32).reshape(1, hkv * G, D)
    kc = kp.ctx.alloc_codes(1, hkv, n)
    for h in range(hkv):
        kp.ctx.quantize(K[0, h], out=tq.Codes(kc.planes[0, h], kc.norm[0, h], kc.signs[0, h], kc.rnorm[0, h]))
    length = torch.tensor([n], dtype=torch.int32, device="cuda")
    scale = 1.0 / sqrt(D)
    out = kp.ctx.attn_output(q, kc, n, length, scale, V).cpu().numpy()
    logits = kp.ctx.attn_logits(q, kc, n, length, scale).cpu().numpy()
    torch.cuda.synchronize()
    assert kp.ctx.sync_status() == 0
    Kc, Vc, qc = K[0].float().cpu().numpy(), V[0].float().cpu().numpy(), q[0].cpu().numpy()
    rng = np.random.default_rng(1)
    for h in (0, 13, 31):
        kvh = h // G
        kz = kp.oquant(Kc[kvh])
        ref_l = scale * oracle.estimate(qc[h], kz, kp.Pi, kp.cb, kp.S)
        ref_o = oracle.turboquant.softmax(ref_l) @ Vc[kvh]
        assert_close(out[0, h], ref_o, "decode-layer output")
        rows = np.sort(rng.choice(n, size=2048, replace=False))
        sel = torch.from_numpy(rows).cuda()
        codes = tq.Codes(planes=kc.planes[0, kvh][sel], norm=kc.norm[0, kvh][sel], signs=kc.signs[0, kvh][sel],
                         rnorm=kc.rnorm[0, kvh][sel])
        same = check_codes(kp, Kc[kvh][rows], codes)
        assert same.mean() > 0.99
        assert_close(logits[0, h, rows][same], ref_l[rows][same], "decode-layer logits")
