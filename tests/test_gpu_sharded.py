"""GPU parity of the sharded attention and search calls (tq_attn_values_partial,
tq_attn_merge_partials, tq_topk_merge) through the C-ABI.  The R blocks of the sequence or of the
database are emulated in one process: each block is scored by the library on its own, the
blocks' partial states or top-k lists are stacked as an all-gather would deliver them, and the
merge is compared with the unsharded oracle.  One more case runs the sharded module itself on a
one-process gloo group."""
import os
import socket
from math import sqrt

import numpy as np
import pytest
import torch

import oracle
from compressed_kv_cache_02_b300 import inputs
from gpu_helpers import Pair, assert_close
from test_gpu_parity import _kv_case, _topk_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")


def _tq():
    from compressed_kv_cache_02_b300 import tq
    return tq


def _block(codes, lo, hi):
    from compressed_kv_cache_02_b300 import tq
    f = lambda t: None if t is None else t[:, :, lo:hi].clone(memory_format=torch.contiguous_format)
    return tq.Codes(planes=f(codes.planes), norm=f(codes.norm), signs=f(codes.signs), rnorm=f(codes.rnorm))


@pytest.mark.parametrize("R", [2, 3])
@pytest.mark.parametrize("vmode", ["mse", "bf16"])
def test_sharded_attention_equals_the_unsharded_oracle(R, vmode):
    tq = _tq()
    from compressed_kv_cache_02_b300 import sharded
    B, Hkv, G, N, d = 2, 2, 4, 1500, 128
    lens = [1500, 400]                     # with R = 3 the second sequence has no keys in two blocks
    c = _kv_case(B, Hkv, G, N, d, 3, vmode, seed=19, lens=lens)
    kp = c["kp"]
    scale = 1.0 / sqrt(d)
    length = torch.tensor(lens, dtype=torch.int32).cuda()
    q = c["q"].cuda()
    parts = []
    for r in range(R):
        lo, hi = sharded.shard_bounds(N, R, r)
        bl = sharded.block_lengths(length, lo, hi)
        logits = kp.ctx.attn_logits(q, _block(c["keys"], lo, hi), hi - lo, bl, scale)
        if vmode == "bf16":
            parts.append(tq.attn_values_partial(logits, bl, c["V"][:, :, lo:hi].contiguous().cuda()))
        else:
            parts.append(tq.attn_values_partial(logits, bl, _block(c["vcodes"], lo, hi), vctx=c["vp"].ctx))
    got = tq.attn_merge_partials(torch.stack(parts), vctx=None if vmode == "bf16" else c["vp"].ctx)
    assert kp.ctx.sync_status() == 0
    if vmode == "bf16":
        ref = oracle.attention_output(c["q"].numpy(), c["kz"], c["lens"], kp.Pi, kp.S, kp.cb, scale,
                                      values_dense=c["V"].float().numpy())
    else:
        vp = c["vp"]
        ref = oracle.attention_output(c["q"].numpy(), c["kz"], c["lens"], kp.Pi, kp.S, kp.cb, scale,
                                      values=c["vz"], Pi_v=vp.Pi, cb_v=vp.cb)
    assert_close(got.cpu().numpy(), ref, f"sharded attention output, {R} blocks")


def test_merge_of_empty_blocks_is_zero():
    tq = _tq()
    d, B, Hq = 128, 1, 4
    parts = torch.zeros(2, B, Hq, d + 2, device="cuda")
    parts[..., 0] = float("-inf")
    out = tq.attn_merge_partials(parts)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


@pytest.mark.parametrize("R,k,bits", [(2, 10, 2), (3, 100, 4), (4, 128, 2)])
def test_sharded_search_equals_the_unsharded_search(R, k, bits):
    tq = _tq()
    from compressed_kv_cache_02_b300 import sharded
    d, n, nq = 200, 3001, 7
    pr = Pair(d, bits, seed=23)
    X = inputs.cone(n, d, seed=23, mu_seed=5)
    X[2900] = X[11]                        # equal codes, hence equal scores, in different blocks
    Q = torch.cat([X[11:12], inputs.cone(nq - 1, d, seed=24, mu_seed=5)])
    z = pr.oquant(X.numpy())
    db = pr.to_device(z, (n,))
    Qd = Q.cuda()
    cs = torch.full((R, nq, k), float("-inf"), device="cuda")
    ci = torch.full((R, nq, k), 2 ** 31 - 1, dtype=torch.int32, device="cuda")
    offs = []
    for r in range(R):
        lo, hi = sharded.shard_bounds(n, R, r)
        # fresh copies: a slice of rows may start off the 16-byte alignment the library requires
        blk = tq.Codes(planes=db.planes[lo:hi].clone(), norm=db.norm[lo:hi].clone(),
                       signs=db.signs[lo:hi].clone(), rnorm=db.rnorm[lo:hi].clone())
        kk = min(k, hi - lo)
        s, i = pr.ctx.search_topk(Qd, blk, kk)
        cs[r, :, :kk] = s
        ci[r, :, :kk] = i
        offs.append(lo)
    got_s, got_i = tq.topk_merge(cs, ci, offs)
    whole_s, whole_i = pr.ctx.search_topk(Qd, db, k)
    assert pr.ctx.sync_status() == 0
    ref_s, ref_i = oracle.search_topk(Q.numpy(), z, pr.Pi, pr.cb, pr.S, k)
    scores = oracle.estimate_all(Q.numpy(), z, pr.Pi, pr.cb, pr.S)
    gs, gi = got_s.cpu().numpy(), got_i.cpu().numpy().astype(np.int64)
    _topk_ok(gs, gi, ref_s, ref_i, scores)
    # every block scores a row exactly as the whole-database search does
    ws, wi = whole_s.cpu().numpy(), whole_i.cpu().numpy().astype(np.int64)
    for r in range(nq):
        common = np.intersect1d(gi[r], wi[r])
        a = {int(i): s for s, i in zip(gs[r], gi[r])}
        b = {int(i): s for s, i in zip(ws[r], wi[r])}
        assert all(a[i] == b[i] for i in common)
    row = list(gi[0])
    assert row.index(11) < row.index(2900)   # the tie across blocks: lower global row first


def test_sharded_module_on_a_one_process_group():
    """compressed_kv_cache_02_b300.sharded with the library's calls on a gloo group of one process
    (the GPU tensors travel through host memory for the all-gather)."""
    import torch.distributed as dist
    from compressed_kv_cache_02_b300 import sharded
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        B, Hkv, G, N, d = 1, 2, 4, 700, 128
        c = _kv_case(B, Hkv, G, N, d, 3, "mse", seed=29, lens=[700])
        kp, vp = c["kp"], c["vp"]
        length = torch.tensor([700], dtype=torch.int32).cuda()
        out = sharded.decode_attention(kp.ctx, c["q"].cuda(), c["keys"], N, length, 1.0 / sqrt(d), c["vcodes"],
                                       vctx=vp.ctx)
        ref = oracle.attention_output(c["q"].numpy(), c["kz"], c["lens"], kp.Pi, kp.S, kp.cb, 1.0 / sqrt(d),
                                      values=c["vz"], Pi_v=vp.Pi, cb_v=vp.cb)
        assert_close(out.cpu().numpy(), ref, "sharded module, one process")
        pr = Pair(200, 2, seed=31)
        X = inputs.cone(500, 200, seed=31, mu_seed=3)
        Q = inputs.cone(4, 200, seed=32, mu_seed=3)
        z = pr.oquant(X.numpy())
        s, i = sharded.search_topk(pr.ctx, Q.cuda(), pr.to_device(z, (500,)), 20, 0)
        ref_s, ref_i = oracle.search_topk(Q.numpy(), z, pr.Pi, pr.cb, pr.S, 20)
        _topk_ok(s.cpu().numpy(), i.cpu().numpy().astype(np.int64), ref_s, ref_i,
                 oracle.estimate_all(Q.numpy(), z, pr.Pi, pr.cb, pr.S))
    finally:
        dist.destroy_process_group()
