"""Host-side pieces of bench.py that need no GPU: the oracle baseline's process pool (one
single-threaded worker per host core, spawned) and its throughput accounting."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def test_oracle_pool_runs_one_group_per_worker():
    import bench
    pool = bench.OraclePool(n_keys=256)
    try:
        assert pool.workers == min(len(os.sched_getaffinity(0)), bench.OraclePool.MAX_WORKERS)
        scores, span, reps, used = pool.run(0.0, 1)
    finally:
        pool.close()
    assert reps == pool.workers                     # one sample per job, one job per worker slot
    assert scores == pool.workers * bench.G * 257   # 4 query heads x (256 cached + 1 appended) keys
    assert span > 0 and 1 <= used <= pool.workers


def test_oracle_sample_scores_the_logits_once():
    import bench
    n, t = bench.oracle_step_sample(128)
    assert n == bench.G * 129 and t > 0
