"""The N > 1 path of bench.py on CPU: two gloo ranks (world size 2, 127.0.0.1) run the
replica helpers the timed region uses — the barrier and the max over ranks of the step time —
and the reference arm, where rank 1 exits without work.  The attention path does not shard
across GPUs in this build (replicas only), so these helpers are the whole multi-process logic."""
import os
import socket
import sys
from types import SimpleNamespace

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    m = bench.max_over_ranks(values[r], w)
    ref = bench.run_reference(SimpleNamespace(steps=1, warmup=0), w, r) if r == 1 else "skipped"
    bench.barrier(w)
    out.put((r, w, m, ref))
    dist.destroy_process_group()


def test_two_gloo_ranks_share_the_max_and_rank1_skips_the_reference_arm():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    values = [1.5, 2.5]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, *_ in res] == [0, 1]
    assert all(w == 2 for _, w, _, _ in res)
    assert all(m == pytest.approx(2.5) for _, _, m, _ in res)   # the timed region takes the slowest rank
    assert res[1][3] is None                                      # rank 1: no oracle work, no line
