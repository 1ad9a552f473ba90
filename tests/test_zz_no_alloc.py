"""tq_attn_values_noalloc: the softmax + value step for callers that cannot allocate device
memory (their memory is pre-reserved or they are given no allocator), using the library's
static scratch array instead of a caller workspace.  Checked through the C-ABI against
tq_attn_values on two calls in a row, within the tolerance of the other GPU tests."""
import numpy as np
import pytest
import torch

from compressed_kv_cache_02_b300 import inputs
from gpu_helpers import ABS, REL

pytestmark = pytest.mark.gpu


def _case(seed, B, Hkv, G, N, d, vctx_codes):
    from compressed_kv_cache_02_b300 import tq
    logits = (inputs.gaussian(B * Hkv * G * N, 1, seed=seed).reshape(B, Hkv * G, N) * 3.0).cuda()
    length = torch.tensor([N - 7 * b for b in range(B)], dtype=torch.int32).cuda()
    if vctx_codes is None:
        fac = inputs.anisotropic_factors(Hkv, d, seed=seed + 1)
        return logits, length, inputs.anisotropic(B, Hkv, N, d, fac, seed=seed + 2).cuda()
    X = inputs.gaussian(B * Hkv * N, d, seed=seed + 3).cuda()
    codes = vctx_codes.quantize(X)
    P = vctx_codes.P
    return logits, length, tq.Codes(planes=codes.planes.reshape(B, Hkv, N, P, -1), norm=codes.norm.reshape(B, Hkv, N))


def _noalloc(tq, vctx, d, logits, length, values):
    B, Hq, cap = logits.shape
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    if vctx is None:
        Hkv, vptr, vnorm, vh = values.shape[1], values.data_ptr(), None, None
    else:
        Hkv, vptr, vnorm, vh = values.planes.shape[1], values.planes.data_ptr(), values.norm.data_ptr(), vctx.h
    rc = tq.lib.tq_attn_values_noalloc(vh, d, logits.data_ptr(), B, Hq, Hkv, cap, length.data_ptr(), vptr, vnorm,
                                      out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == tq.TQ_OK, tq.lib.tq_last_error()
    return out


def _close(a, b):
    a, b = a.cpu().double().numpy(), b.cpu().double().numpy()
    err = np.abs(a - b)
    assert np.all((err <= ABS) | (err <= REL * np.abs(b)))


@pytest.mark.parametrize("coded", [False, True])
def test_noalloc_matches_workspace_entry_twice(coded):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from compressed_kv_cache_02_b300 import tq
    d = 128
    vctx = tq.Context(d, 3, seed=5, mode=tq.TQ_MODE_MSE) if coded else None
    for call, (B, Hkv, G, N) in enumerate([(2, 4, 4, 3000), (1, 8, 4, 777)]):   # two calls in a row
        logits, length, values = _case(40 + call, B, Hkv, G, N, d, vctx)
        ref = tq.attn_values(logits, length, values, vctx=vctx)
        got = _noalloc(tq, vctx, d, logits, length, values)
        torch.cuda.synchronize()
        _close(got, ref)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from compressed_kv_cache_02_b300 import tq
    B, Hq, Hkv, d, cap = 64, 64, 8, 512, 1 << 20
    need = tq._sz()
    assert tq.lib.tq_attn_values_workspace_size(d, B, Hq, Hkv, cap, need) == tq.TQ_OK
    assert need.value > (8 << 20)
    dummy = torch.zeros(64, device="cuda")
    rc = tq.lib.tq_attn_values_noalloc(None, d, dummy.data_ptr(), B, Hq, Hkv, cap, dummy.data_ptr(),
                                      dummy.data_ptr(), None, dummy.data_ptr(), None)
    assert rc == tq.TQ_ERR_UNSUPPORTED
    assert b"static array" in tq.lib.tq_last_error()
