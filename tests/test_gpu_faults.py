"""Host-side fault injection on a GPU machine: a simulated out-of-memory at every allocation point of
tq_init_ex returns TQ_ERR_OOM with a NULL context and frees what was allocated (100 failures at
the last allocation leave the free device memory unchanged); afterwards contexts work normally."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import Pair, check_codes

pytestmark = pytest.mark.gpu


def _tq():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from compressed_kv_cache_02_b300 import tq
    return tq


def _init(tq):
    h = ctypes.c_void_p()
    rc = tq.lib.tq_init_ex(ctypes.byref(h), 0, 128, 3, tq.TQ_MODE_PROD, 128, None, None)
    return rc, h


def test_simulated_allocation_failures_free_everything():
    tq = _tq()
    try:
        allocs = 0
        for n in range(32):   # fail allocation n + 1 until init needs fewer
            assert tq.lib.tq_debug_fail_alloc_after(n) == tq.TQ_OK
            rc, h = _init(tq)
            if rc == tq.TQ_OK:
                tq.lib.tq_destroy(h)
                allocs = n
                break
            assert rc == tq.TQ_ERR_OOM and not h.value
            assert b"simulated" in tq.lib.tq_last_error()
        assert allocs >= 4   # matrices, JL operands, error word at least
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for _ in range(100):   # the last allocation fails: everything before it must be freed
            tq.lib.tq_debug_fail_alloc_after(allocs - 1)
            rc, h = _init(tq)
            assert rc == tq.TQ_ERR_OOM and not h.value
        torch.cuda.synchronize()
        assert free0 - torch.cuda.mem_get_info()[0] < (16 << 20)
    finally:
        tq.lib.tq_debug_fail_alloc_after(-1)
    kp = Pair(128, 3, seed=0)
    x = torch.randn(16, 128).cuda()
    codes = kp.ctx.quantize(x)
    assert kp.ctx.sync_status() == 0
    check_codes(kp, x.cpu().numpy(), codes)
