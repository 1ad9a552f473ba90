"""The multi-process (sharded) attention and search of compressed_kv_cache_02_b300.sharded on CPU:
two and three gloo ranks (127.0.0.1) each hold a block of the sequence or of the database.  The
module's host logic runs as written -- block bounds and lengths, padding of short blocks, the
all-gathers and their rank order, the row offsets -- while the device work is done by the oracle
(passed as the `ops` object), so the merged results can be compared with the unsharded oracle."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """The device steps of the sharded module done by the oracle on CPU tensors (test only)."""

    score_dtype = torch.float64

    def __init__(self, Hkv):
        self.Hkv = Hkv

    def rows(self, db):
        return int(db.idx.shape[0])

    def logits(self, kctx, q, keys, cap, length, scale):
        import oracle
        Pi, S, cb = kctx
        lg = oracle.attention_logits(q.numpy(), keys, length.numpy(), Pi, S, cb, scale)
        return torch.from_numpy(np.nan_to_num(lg, nan=0.0))

    def values_partial(self, logits, length, values, vctx):
        from oracle import sharded as osh
        Piv, cbv = vctx
        m, l, a = osh.attention_partial(logits.numpy(), length.numpy(), self.Hkv, values=values, cb_v=cbv)
        return torch.from_numpy(np.concatenate([m[..., None], l[..., None], a], axis=-1))

    def merge_partials(self, parts, vctx):
        from oracle import sharded as osh
        Piv, _ = vctx
        p = parts.numpy()
        return torch.from_numpy(osh.merge_partials([(p[r, ..., 0], p[r, ..., 1], p[r, ..., 2:]) for r in range(p.shape[0])],
                                                   Piv))

    def search_topk(self, ctx, q, db, k):
        import oracle
        Pi, S, cb = ctx
        s, i = oracle.search_topk(q.numpy(), db, Pi, cb, S, k)
        return torch.from_numpy(s), torch.from_numpy(i)

    def topk_merge(self, cand_s, cand_i, row_offsets):
        from oracle import sharded as osh
        lists = []
        for r, off in enumerate(row_offsets):
            i = cand_i[r].numpy().astype(np.int64)
            lists.append((cand_s[r].numpy(), np.where(i == 2 ** 31 - 1, np.iinfo(np.int64).max, i + off)))
        s, i = osh.merge_topk(lists, cand_s.shape[2])
        return torch.from_numpy(s), torch.from_numpy(i)


def _problem():
    import oracle
    from oracle import rng
    B, Hkv, G, N, d = 2, 2, 4, 37, 16
    Pi, S = rng.method_matrices(3, d, d)
    Piv, _ = rng.method_matrices(4, d, 1)
    cbk, cbv = oracle.sphere_codebook(d, 2), oracle.sphere_codebook(d, 3)
    K = rng.gaussian_stream(5, B * Hkv * N * d).reshape(B, Hkv, N, d)
    V = rng.gaussian_stream(6, B * Hkv * N * d).reshape(B, Hkv, N, d)
    q = rng.gaussian_stream(7, B * Hkv * G * d).reshape(B, Hkv * G, d)
    kz, vz = oracle.quantize(K, Pi, cbk, S), oracle.quantize(V, Piv, cbv)
    lens = np.array([N, 20])
    n, nq = 101, 5
    X = rng.gaussian_stream(8, n * d).reshape(n, d)
    Q = rng.gaussian_stream(9, nq * d).reshape(nq, d)
    dz = oracle.quantize(X, Pi, cbk, S)
    return dict(B=B, Hkv=Hkv, N=N, d=d, Pi=Pi, S=S, Piv=Piv, cbk=cbk, cbv=cbv, q=q, kz=kz, vz=vz, lens=lens,
                n=n, Q=Q, dz=dz)


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    from compressed_kv_cache_02_b300 import sharded
    dist.init_process_group("gloo", rank=rank, world_size=world)
    p = _problem()
    ops = OracleOps(p["Hkv"])
    # attention: this rank's block of every sequence
    lo, hi = sharded.shard_bounds(p["N"], world, rank)
    blk = lambda z, signs: oracle.Quantized(
        idx=z.idx[:, :, lo:hi], norm16=z.norm16[:, :, lo:hi],
        signs=z.signs[:, :, lo:hi] if signs else None, rnorm16=z.rnorm16[:, :, lo:hi] if signs else None)
    length = sharded.block_lengths(torch.from_numpy(p["lens"]), lo, hi)
    o = sharded.decode_attention((p["Pi"], p["S"], p["cbk"]), torch.from_numpy(p["q"]), blk(p["kz"], True), hi - lo,
                                 length, 1.0 / 4.0, blk(p["vz"], False), vctx=(p["Piv"], p["cbv"]), ops=ops)
    # search: this rank's block of the database
    lo, hi = sharded.shard_bounds(p["n"], world, rank)
    z = p["dz"]
    db = oracle.Quantized(idx=z.idx[lo:hi], norm16=z.norm16[lo:hi], signs=z.signs[lo:hi], rnorm16=z.rnorm16[lo:hi])
    k = 40 if world == 3 else 60          # 60 > a block of 50 rows: the short block is padded
    s, i = sharded.search_topk((p["Pi"], p["S"], p["cbk"]), torch.from_numpy(p["Q"]), db, k, lo, ops=ops)
    out.put((rank, o.numpy(), s.numpy(), i.numpy(), k))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_attention_and_search_equal_the_unsharded_oracle(world):
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    pb = _problem()
    logits = oracle.attention_logits(pb["q"], pb["kz"], pb["lens"], pb["Pi"], pb["S"], pb["cbk"], 1.0 / 4.0)
    ref = oracle.attention_values(np.nan_to_num(logits, nan=0.0), pb["lens"], pb["Hkv"], values=pb["vz"],
                                  Pi_v=pb["Piv"], cb_v=pb["cbv"])
    k = res[0][4]
    ref_s, ref_i = oracle.search_topk(pb["Q"], pb["dz"], pb["Pi"], pb["cbk"], pb["S"], k)
    all_s = oracle.estimate_all(pb["Q"], pb["dz"], pb["Pi"], pb["cbk"], pb["S"])
    for rank, o, s, i, _ in res:                       # every rank holds the whole result
        assert np.max(np.abs(o - ref)) < 1e-12
        assert np.max(np.abs(s - ref_s)) < 1e-12 * np.max(np.abs(ref_s))
        for r in range(i.shape[0]):
            for a, b in zip(i[r], ref_i[r]):
                if a != b:                            # float64 near-ties may trade places
                    assert abs(all_s[r, a] - all_s[r, b]) < 1e-12 * abs(all_s[r, b])
