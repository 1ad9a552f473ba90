"""CPU-side checks of libtq: it loads, exports every symbol of include/tq.h, and its host
set-up (codebook by Gauss-Legendre quadrature, seeded matrices by its own C++ generator)
agrees with the oracle's independent computations.  No GPU needed."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from oracle.codebook import sphere_codebook

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tq.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def tq():
    from compressed_kv_cache_02_b300 import build
    build.build()
    from compressed_kv_cache_02_b300 import tq as mod
    return mod


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("tq_init", "tq_quantize", "tq_attn_logits", "tq_attn_output", "tq_search_topk"):
        assert required in names


def test_library_exports_every_declared_symbol(tq):
    missing = [n for n in _declared_functions() if not hasattr(tq.lib, n)]
    assert missing == []


@pytest.mark.parametrize("d", [3, 16, 128, 200, 1024])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_host_codebook_matches_oracle(tq, d, bits):
    c, t = tq.host_codebook(d, bits)
    ref = sphere_codebook(d, bits)
    assert np.max(np.abs(c - ref.centroids)) < 1e-12
    assert np.max(np.abs(t - ref.thresholds)) < 1e-12


@pytest.mark.parametrize("d", [3, 16, 128, 200, 1024])
@pytest.mark.parametrize("bits", [5, 6, 7, 8])
def test_host_codebook_wide_matches_oracle(tq, d, bits):
    # From 5 bits both sides solve the Lloyd-Max conditions by Newton's method, each with its own
    # quadrature (library: composite Gauss-Legendre; oracle: incomplete beta).  The fixed point is
    # then determined only to ~L^2 times the rounding of one Lloyd step (the smallest eigenvalue of
    # the step's Jacobian is ~(pi/L)^2), so the two tables agree to that level, far below the
    # float32 rounding the kernels apply, and the library's table passes the oracle's own Lloyd
    # step to that step's rounding floor.
    from oracle import codebook as cbm
    c, t = tq.host_codebook(d, bits)
    ref = sphere_codebook(d, bits)
    tol = 2e-12 * 4.0 ** (bits - 4)
    assert np.max(np.abs(c - ref.centroids)) < tol
    assert np.max(np.abs(t - ref.thresholds)) < tol
    _, _, _, _, g = cbm._cells(c, d)
    assert np.max(np.abs(g - c)) < 2e-13
    assert np.array_equal(c, -c[::-1]) and np.all(np.diff(c) > 0)


@pytest.mark.parametrize("d,m", [(4, 4), (16, 16), (128, 128), (200, 200), (40, 24)])
def test_host_matrices_match_oracle_generator(tq, d, m):
    Pi, S = tq.host_matrices(7, d, m)
    Pi_o, S_o = oracle.method_matrices(7, d, m)
    assert np.array_equal(S, S_o.astype(np.float32))
    # both QRs give the same Haar matrix up to float64 rounding, then one float32 rounding
    assert np.max(np.abs(Pi.astype(np.float64) - Pi_o)) < 2 ** -23
    assert np.max(np.abs(Pi.astype(np.float64).T @ Pi - np.eye(d))) < 1e-5


def test_host_argument_errors(tq):
    c = np.zeros(2)
    assert tq.lib.tq_host_codebook(2, 1, c.ctypes.data, None) == tq.TQ_ERR_ARG
    assert tq.lib.tq_host_codebook(128, 9, c.ctypes.data, None) == tq.TQ_ERR_ARG
    assert b"mse_bits" in tq.lib.tq_last_error()
    assert tq.lib.tq_host_matrices(0, 2000, 4, None, None) == tq.TQ_ERR_ARG


def test_context_calls_reject_null_context(tq):
    assert tq.lib.tq_quantize(None, None, 0, 1, 1, None, None, None, None, None) == tq.TQ_ERR_ARG
    assert tq.lib.tq_info(None, None, None, None, None) == tq.TQ_ERR_ARG
    tq.lib.tq_destroy(None)   # no-op


@pytest.mark.parametrize("level", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_host_polar_codebook_matches_oracle(tq, level, bits):
    c, t = tq.host_polar_codebook(level, bits)
    ref = oracle.angle_codebook(level, bits)
    assert np.max(np.abs(c - ref.centroids)) < 1e-11
    assert np.max(np.abs(t - ref.thresholds)) < 1e-11


def test_polar_calls_reject_bad_arguments(tq):
    import ctypes
    c, t = np.zeros(16), np.zeros(15)
    assert tq.lib.tq_host_polar_codebook(0, 2, c.ctypes.data, t.ctypes.data) == tq.TQ_ERR_ARG
    assert tq.lib.tq_host_polar_codebook(2, 5, c.ctypes.data, t.ctypes.data) == tq.TQ_ERR_ARG
    h = ctypes.c_void_p()
    assert tq.lib.tq_polar_init(ctypes.byref(h), 0, 100, 3, 1, None, None) == tq.TQ_ERR_ARG   # not a power of two
    assert tq.lib.tq_polar_init(ctypes.byref(h), 0, 8, 3, 1, None, None) == tq.TQ_ERR_ARG     # below 16
    assert tq.lib.tq_polar_init(ctypes.byref(h), 0, 128, 5, 1, None, None) == tq.TQ_ERR_ARG   # bits
    assert tq.lib.tq_polar_init(ctypes.byref(h), 0, 128, 3, 2, None, None) == tq.TQ_ERR_ARG   # qjl flag
    assert tq.lib.tq_polar_quantize(None, None, 0, 1, 128, None, None, None, None, None) == tq.TQ_ERR_ARG
    assert tq.lib.tq_polar_scores(None, None, 1, None, None, None, None, 1, 1.0, None, None) == tq.TQ_ERR_ARG
    assert tq.lib.tq_polar_layout(None, None, None) == tq.TQ_ERR_ARG
    tq.lib.tq_polar_destroy(None)   # no-op


def test_paged_calls_reject_bad_arguments(tq):
    import ctypes
    n = ctypes.c_size_t()
    assert tq.lib.tq_paged_workspace_size(2, 8, 2, 4, 48, ctypes.byref(n)) == tq.TQ_ERR_ARG   # page_size % 32
    assert tq.lib.tq_paged_workspace_size(2, 7, 2, 4, 64, ctypes.byref(n)) == tq.TQ_ERR_ARG   # Hq % Hkv
    assert tq.lib.tq_paged_workspace_size(2, 8, 2, 4, 64, ctypes.byref(n)) == tq.TQ_OK and n.value > 0
    assert tq.lib.tq_paged_decode_step(None, None, *([None] * 3), 0, 1, 4, 1, None, 1, 32, 1, None,
                                       *([None] * 6), 1.0, None, None, 0, None) == tq.TQ_ERR_ARG


def test_alloc_fault_hook_rejects_bad_values(tq):
    assert tq.lib.tq_debug_fail_alloc_after(-2) == tq.TQ_ERR_ARG
    assert tq.lib.tq_debug_fail_alloc_after(-1) == tq.TQ_OK
