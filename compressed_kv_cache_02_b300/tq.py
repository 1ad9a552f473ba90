"""Thin ctypes binding of libtq (include/tq.h): argument marshalling only.

Every compute call passes device pointers of caller-owned torch tensors and the current
CUDA stream to the C-ABI; all arithmetic happens in the library's kernels.  Importing
this module loads ``libtq.so`` from this package directory and raises if it is missing:
there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtq.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libtq.so not found at {_LIB_PATH}; build it with "
                      "`python -m compressed_kv_cache_02_b300.build`")
lib = ctypes.CDLL(_LIB_PATH)

TQ_OK, TQ_ERR_ARG, TQ_ERR_CUDA, TQ_ERR_OOM, TQ_ERR_UNSUPPORTED, TQ_ERR_DEVICE = range(6)
TQ_F32, TQ_BF16 = 0, 1
TQ_MODE_PROD, TQ_MODE_MSE = 0, 1
TQ_MAX_TOPK = 128
TQ_DEVERR_NORM_OVERFLOW, TQ_DEVERR_LEN_RANGE, TQ_DEVERR_TIMEOUT = 1, 2, 4
TQ_PATH_AUTO, TQ_PATH_CUDA_CORE, TQ_PATH_TENSOR = 0, 1, 2

_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_f = ctypes.c_float
_sz = ctypes.c_size_t

_SIGS = {
    "tq_host_codebook": [_i, _i, _p, _p],
    "tq_host_matrices": [_u64, _i, _i, _p, _p],
    "tq_init": [ctypes.POINTER(_p), _u64, _i, _i],
    "tq_init_ex": [ctypes.POINTER(_p), _u64, _i, _i, _i, _i, _p, _p],
    "tq_init_split": [ctypes.POINTER(_p), _u64, _i, _i, _i, _i, _i, _p, _p],
    "tq_code_words": [_p, _p, _p],
    "tq_info": [_p, _p, _p, _p, _p],
    "tq_layout": [_p, _p, _p, _p],
    "tq_export_matrices": [_p, _p, _p, _p, _p],
    "tq_set_kernel_path": [_p, _i],
    "tq_quantize": [_p, _p, _i, _i64, _i64, _p, _p, _p, _p, _p],
    "tq_append": [_p, _p, _i, _i, _i, _i64, _p, _p, _p, _p, _p, _p],
    "tq_advance_len": [_p, _p, _i, _i64, _i, _p],
    "tq_prep_queries": [_p, _p, _i64, _p, _p, _p],
    "tq_attn_workspace_size": [_p, _i, _i, _i, _i64, ctypes.POINTER(_sz)],
    "tq_attn_logits": [_p, _p, _i, _i, _i, _p, _p, _p, _p, _i64, _p, _f, _p, _p, _sz, _p],
    "tq_attn_output": [_p, _p, _p, _i, _i, _i, _p, _p, _p, _p, _i64, _p, _f, _p, _p, _p, _p, _sz, _p],
    "tq_attn_values_workspace_size": [_i, _i, _i, _i, _i64, ctypes.POINTER(_sz)],
    "tq_attn_values": [_p, _i, _p, _i, _i, _i, _i64, _p, _p, _p, _p, _p, _sz, _p],
    "tq_attn_values_noalloc": [_p, _i, _p, _i, _i, _i, _i64, _p, _p, _p, _p, _p],
    "tq_attn_values_partial": [_p, _i, _p, _i, _i, _i, _i64, _p, _p, _p, _p, _p, _sz, _p],
    "tq_attn_merge_partials": [_p, _i, _p, _i, _i, _i, _p, _p],
    "tq_topk_merge": [_p, _p, _i, _i64, _i, _p, _p, _p, _p],
    "tq_search_workspace_size": [_p, _i64, _i64, _i, ctypes.POINTER(_sz)],
    "tq_search_topk": [_p, _p, _i64, _p, _p, _p, _p, _i64, _i, _p, _p, _p, _sz, _p],
    "tq_sync_status": [_p, _p, _p],
    "tq_host_polar_codebook": [_i, _i, _p, _p],
    "tq_polar_init": [ctypes.POINTER(_p), _u64, _i, _i, _i, _p, _p],
    "tq_polar_layout": [_p, _p, _p],
    "tq_polar_quantize": [_p, _p, _i, _i64, _i64, _p, _p, _p, _p, _p],
    "tq_polar_set_kernel_path": [_p, _i],
    "tq_polar_scores": [_p, _p, _i64, _p, _p, _p, _p, _i64, _f, _p, _p],
    "tq_polar_sync_status": [_p, _p, _p],
    "tq_paged_workspace_size": [_i, _i, _i, _i, _i, ctypes.POINTER(_sz)],
    "tq_selftest_wait_timeout": [_p, _p],
    "tq_debug_fail_alloc_after": [_i],
    "tq_paged_decode_step": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _p, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _f, _p,
                             _p, _sz, _p],
}
for _name, _args in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = _i
lib.tq_destroy.argtypes = [_p]
lib.tq_destroy.restype = None
lib.tq_polar_destroy.argtypes = [_p]
lib.tq_polar_destroy.restype = None
lib.tq_last_error.argtypes = []
lib.tq_last_error.restype = ctypes.c_char_p


class TQError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where} failed with status {code}: {lib.tq_last_error().decode()}")


def _check(code: int, where: str) -> None:
    if code != TQ_OK:
        raise TQError(code, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr() if t.numel() else None
    return t


def _stream(stream=None):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def host_codebook(d: int, mse_bits: int):
    import numpy as np
    c = np.zeros(1 << mse_bits)
    t = np.zeros((1 << mse_bits) - 1)
    _check(lib.tq_host_codebook(d, mse_bits, c.ctypes.data, t.ctypes.data if t.size else None), "tq_host_codebook")
    return c, t


def host_matrices(seed: int, d: int, m: int):
    import numpy as np
    Pi = np.zeros((d, d), dtype=np.float32)
    S = np.zeros((m, d), dtype=np.float32)
    _check(lib.tq_host_matrices(seed, d, m, Pi.ctypes.data, S.ctypes.data), "tq_host_matrices")
    return Pi, S


@dataclass
class Codes:
    """Packed codes of a batch of vectors (device tensors, layout of include/tq.h)."""
    planes: torch.Tensor
    norm: torch.Tensor
    signs: torch.Tensor | None = None
    rnorm: torch.Tensor | None = None


def values_workspace(d, B, Hq, Hkv, cap, device="cuda") -> torch.Tensor:
    n = _sz()
    _check(lib.tq_attn_values_workspace_size(d, B, Hq, Hkv, cap, ctypes.byref(n)), "tq_attn_values_workspace_size")
    return torch.empty(n.value, dtype=torch.uint8, device=device)


def attn_values(logits, length, values, vctx=None, d=None, Hkv=None, out=None, workspace=None, stream=None):
    """Softmax over logits [B, Hq, cap] and the weighted sum of values: bf16 [B, Hkv, cap, d]
    (vctx None) or the Codes of an MSE-mode vctx."""
    B, Hq, cap = logits.shape
    if vctx is None:
        Hkv, d = values.shape[1], values.shape[3]
        vptr, vnorm, vh = _ptr(values), None, None
    else:
        Hkv, d = values.planes.shape[1], vctx.d
        vptr, vnorm, vh = _ptr(values.planes), _ptr(values.norm), vctx.h
    if out is None:
        out = torch.empty(B, Hq, d, device=logits.device, dtype=torch.float32)
    if workspace is None:
        workspace = values_workspace(d, B, Hq, Hkv, cap, device=logits.device)
    _check(lib.tq_attn_values(vh, d, _ptr(logits), B, Hq, Hkv, cap, _ptr(length), vptr, vnorm, _ptr(out),
                              _ptr(workspace), workspace.numel(), _stream(stream)), "tq_attn_values")
    return out


def attn_values_partial(logits, length, values, vctx=None, out=None, workspace=None, stream=None):
    """tq_attn_values_partial: this block's partial states [B, Hq, d + 2] = (max, weight sum,
    weighted value sum) over logits [B, Hq, cap] and its values (bf16 [B, Hkv, cap, d] or Codes)."""
    B, Hq, cap = logits.shape
    if vctx is None:
        Hkv, d = values.shape[1], values.shape[3]
        vptr, vnorm, vh = _ptr(values), None, None
    else:
        Hkv, d = values.planes.shape[1], vctx.d
        vptr, vnorm, vh = _ptr(values.planes), _ptr(values.norm), vctx.h
    if out is None:
        out = torch.empty(B, Hq, d + 2, device=logits.device, dtype=torch.float32)
    if workspace is None:
        workspace = values_workspace(d, B, Hq, Hkv, cap, device=logits.device)
    _check(lib.tq_attn_values_partial(vh, d, _ptr(logits), B, Hq, Hkv, cap, _ptr(length), vptr, vnorm, _ptr(out),
                                      _ptr(workspace), workspace.numel(), _stream(stream)), "tq_attn_values_partial")
    return out


def attn_merge_partials(parts, vctx=None, out=None, stream=None):
    """tq_attn_merge_partials: parts [R, B, Hq, d + 2] of R blocks -> out [B, Hq, d]."""
    R, B, Hq, d2 = parts.shape
    d = d2 - 2
    parts = parts.contiguous()
    if out is None:
        out = torch.empty(B, Hq, d, device=parts.device, dtype=torch.float32)
    _check(lib.tq_attn_merge_partials(None if vctx is None else vctx.h, d, _ptr(parts), R, B, Hq, _ptr(out),
                                      _stream(stream)), "tq_attn_merge_partials")
    return out


def topk_merge(cand_s, cand_i, row_offsets, stream=None):
    """tq_topk_merge: R blocks' lists cand_s / cand_i [R, nq, k] (block-local rows, INT32_MAX =
    padding) and their first global rows -> global top_s, top_i [nq, k]."""
    import numpy as np
    R, nq, k = cand_s.shape
    offs = np.ascontiguousarray(np.asarray(row_offsets, dtype=np.int64))
    top_s = torch.empty(nq, k, device=cand_s.device, dtype=torch.float32)
    top_i = torch.empty(nq, k, device=cand_s.device, dtype=torch.int32)
    _check(lib.tq_topk_merge(_ptr(cand_s.contiguous()), _ptr(cand_i.contiguous()), R, nq, k, offs.ctypes.data,
                             _ptr(top_s), _ptr(top_i), _stream(stream)), "tq_topk_merge")
    return top_s, top_i


class Context:
    """A tq_ctx: seeded rotation, JL matrix and codebook on the current device."""

    def __init__(self, d: int, bits: int, seed: int = 0, mode: int = TQ_MODE_PROD, m: int | None = None,
                 Pi=None, S=None, d_hi: int = 0):
        """d_hi > 0: split (fractional bit width) context, see tq_init_split."""
        import numpy as np
        h = _p()
        Pi_a = None if Pi is None else np.ascontiguousarray(Pi, dtype=np.float32)
        S_a = None if S is None else np.ascontiguousarray(S, dtype=np.float32)
        if m is None:
            m = d
        _check(lib.tq_init_split(ctypes.byref(h), seed, d, bits, d_hi, mode, m,
                                 None if Pi_a is None else Pi_a.ctypes.data,
                                 None if S_a is None else S_a.ctypes.data), "tq_init_split")
        self.h = h
        d_, m_, p_, mode_ = _i(), _i(), _i(), _i()
        _check(lib.tq_info(h, ctypes.byref(d_), ctypes.byref(m_), ctypes.byref(p_), ctypes.byref(mode_)), "tq_info")
        self.d, self.m, self.P, self.mode = d_.value, m_.value, p_.value, mode_.value
        w, ws = _i(), _i()
        _check(lib.tq_layout(h, None, ctypes.byref(w), ctypes.byref(ws)), "tq_layout")
        self.W, self.Ws = w.value, ws.value
        rw, dh = _i(), _i()
        _check(lib.tq_code_words(h, ctypes.byref(rw), ctypes.byref(dh)), "tq_code_words")
        self.row_words, self.d_hi = rw.value, dh.value

    def close(self):
        if getattr(self, "h", None):
            lib.tq_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def qjl(self) -> bool:
        return self.mode == TQ_MODE_PROD

    def set_kernel_path(self, path: int) -> None:
        _check(lib.tq_set_kernel_path(self.h, path), "tq_set_kernel_path")

    def export(self):
        import numpy as np
        Pi = np.zeros((self.d, self.d), dtype=np.float32)
        S = np.zeros((max(self.m, 1), self.d), dtype=np.float32)
        c = np.zeros(1 << self.P)
        t = np.zeros((1 << self.P) - 1)
        _check(lib.tq_export_matrices(self.h, Pi.ctypes.data, S.ctypes.data if self.m else None, c.ctypes.data,
                                      t.ctypes.data if t.size else None), "tq_export_matrices")
        return Pi, (S if self.m else None), c, t

    def alloc_codes(self, *shape, device="cuda") -> Codes:
        """Zeroed code buffers for rows of the given leading shape (planes [..., P, W]; a split
        context's rows are flat [..., row_words])."""
        if self.d_hi:
            planes = torch.zeros(*shape, self.row_words, dtype=torch.int32, device=device)
        else:
            planes = torch.zeros(*shape, self.P, self.W, dtype=torch.int32, device=device)
        norm = torch.zeros(*shape, dtype=torch.int16, device=device)
        if not self.qjl:
            return Codes(planes=planes, norm=norm)
        signs = torch.zeros(*shape, self.Ws, dtype=torch.int32, device=device)
        rnorm = torch.zeros(*shape, dtype=torch.int16, device=device)
        return Codes(planes=planes, norm=norm, signs=signs, rnorm=rnorm)

    # -- calls (names follow the C-ABI) ---------------------------------------------------
    def quantize(self, x: torch.Tensor, out: Codes | None = None, stream=None) -> Codes:
        x2 = x.reshape(-1, self.d)
        if out is None:
            out = self.alloc_codes(x2.shape[0], device=x.device)
        dtype = TQ_BF16 if x.dtype == torch.bfloat16 else TQ_F32
        if x.dtype not in (torch.bfloat16, torch.float32):
            raise TypeError("x must be float32 or bfloat16")
        _check(lib.tq_quantize(self.h, _ptr(x2), dtype, x2.shape[0], x2.stride(0), _ptr(out.planes), _ptr(out.signs),
                               _ptr(out.norm), _ptr(out.rnorm), _stream(stream)), "tq_quantize")
        return out

    def append(self, x: torch.Tensor, cache: Codes, cap: int, length: torch.Tensor, stream=None) -> None:
        B, H, d = x.shape
        dtype = TQ_BF16 if x.dtype == torch.bfloat16 else TQ_F32
        _check(lib.tq_append(self.h, _ptr(x.contiguous()), dtype, B, H, cap, _ptr(length), _ptr(cache.planes),
                             _ptr(cache.signs), _ptr(cache.norm), _ptr(cache.rnorm), _stream(stream)), "tq_append")

    def advance_len(self, length: torch.Tensor, cap: int, step: int = 1, stream=None) -> None:
        _check(lib.tq_advance_len(self.h, _ptr(length), length.numel(), cap, step, _stream(stream)), "tq_advance_len")

    def prep_queries(self, q: torch.Tensor, stream=None):
        q2 = q.reshape(-1, self.d).contiguous()
        qrot = torch.empty_like(q2)
        qproj = torch.empty(q2.shape[0], self.m, device=q.device, dtype=torch.float32) if self.qjl else None
        _check(lib.tq_prep_queries(self.h, _ptr(q2), q2.shape[0], _ptr(qrot), _ptr(qproj), _stream(stream)),
               "tq_prep_queries")
        return qrot, qproj

    def attn_workspace(self, B, Hq, Hkv, cap, device="cuda") -> torch.Tensor:
        n = _sz()
        _check(lib.tq_attn_workspace_size(self.h, B, Hq, Hkv, cap, ctypes.byref(n)), "tq_attn_workspace_size")
        return torch.empty(n.value, dtype=torch.uint8, device=device)

    def attn_logits(self, q, keys: Codes, cap, length, scale, out=None, workspace=None, stream=None):
        B, Hq, d = q.shape
        Hkv = keys.planes.shape[1]
        if out is None:
            out = torch.empty(B, Hq, cap, device=q.device, dtype=torch.float32)
        if workspace is None:
            workspace = self.attn_workspace(B, Hq, Hkv, cap, device=q.device)
        _check(lib.tq_attn_logits(self.h, _ptr(q), B, Hq, Hkv, _ptr(keys.planes), _ptr(keys.signs), _ptr(keys.norm),
                                  _ptr(keys.rnorm), cap, _ptr(length), float(scale), _ptr(out), _ptr(workspace),
                                  workspace.numel(), _stream(stream)), "tq_attn_logits")
        return out

    def attn_output(self, q, keys: Codes, cap, length, scale, values, vctx: "Context | None" = None,
                    out=None, workspace=None, stream=None):
        """values: a bf16 tensor [B, Hkv, cap, d] (vctx None) or Codes of an MSE-mode vctx."""
        B, Hq, d = q.shape
        Hkv = keys.planes.shape[1]
        if out is None:
            out = torch.empty(B, Hq, d, device=q.device, dtype=torch.float32)
        if workspace is None:
            workspace = self.attn_workspace(B, Hq, Hkv, cap, device=q.device)
        if vctx is None:
            vptr, vnorm = _ptr(values), None
        else:
            vptr, vnorm = _ptr(values.planes), _ptr(values.norm)
        _check(lib.tq_attn_output(self.h, None if vctx is None else vctx.h, _ptr(q), B, Hq, Hkv, _ptr(keys.planes),
                                  _ptr(keys.signs), _ptr(keys.norm), _ptr(keys.rnorm), cap, _ptr(length),
                                  float(scale), vptr, vnorm, _ptr(out), _ptr(workspace), workspace.numel(),
                                  _stream(stream)), "tq_attn_output")
        return out

    def search_workspace(self, nq, n, k, device="cuda") -> torch.Tensor:
        s = _sz()
        _check(lib.tq_search_workspace_size(self.h, nq, n, k, ctypes.byref(s)), "tq_search_workspace_size")
        return torch.empty(s.value, dtype=torch.uint8, device=device)

    def search_topk(self, q, db: Codes, k, workspace=None, stream=None):
        nq = q.shape[0]
        n = db.planes.shape[0]
        scores = torch.empty(nq, k, device=q.device, dtype=torch.float32)
        idx = torch.empty(nq, k, device=q.device, dtype=torch.int32)
        if workspace is None:
            workspace = self.search_workspace(nq, n, k, device=q.device)
        _check(lib.tq_search_topk(self.h, _ptr(q), nq, _ptr(db.planes), _ptr(db.signs), _ptr(db.norm),
                                  _ptr(db.rnorm), n, k, _ptr(scores), _ptr(idx), _ptr(workspace), workspace.numel(),
                                  _stream(stream)), "tq_search_topk")
        return scores, idx

    def sync_status(self, stream=None) -> int:
        flags = _i(0)
        code = lib.tq_sync_status(self.h, _stream(stream), ctypes.byref(flags))
        if code not in (TQ_OK, TQ_ERR_DEVICE):
            raise TQError(code, "tq_sync_status")
        return flags.value


# ---------------------------------------------------------------------------------- polar encoder

def host_polar_codebook(level: int, bits: int):
    import numpy as np
    c = np.zeros(1 << bits)
    t = np.zeros((1 << bits) - 1)
    _check(lib.tq_host_polar_codebook(level, bits, c.ctypes.data, t.ctypes.data if t.size else None),
           "tq_host_polar_codebook")
    return c, t


@dataclass
class PolarCodes:
    """Packed polar codes of a batch of vectors (device tensors, layout of include/tq.h)."""
    codes: torch.Tensor
    r16: torch.Tensor
    signs: torch.Tensor | None = None
    rnorm: torch.Tensor | None = None


class PolarContext:
    """A tq_polar: seeded rotation (and JL matrix), per-level angle tables on the current device."""

    def __init__(self, d: int, bits: int, qjl: bool = True, seed: int = 0, Pi=None, S=None):
        import numpy as np
        h = _p()
        Pi_a = None if Pi is None else np.ascontiguousarray(Pi, dtype=np.float32)
        S_a = None if S is None else np.ascontiguousarray(S, dtype=np.float32)
        _check(lib.tq_polar_init(ctypes.byref(h), seed, d, bits, int(qjl),
                                 None if Pi_a is None else Pi_a.ctypes.data,
                                 None if S_a is None else S_a.ctypes.data), "tq_polar_init")
        self.h, self.d, self.bits, self.qjl = h, d, bits, bool(qjl)
        cw, ws = _i(), _i()
        _check(lib.tq_polar_layout(h, ctypes.byref(cw), ctypes.byref(ws)), "tq_polar_layout")
        self.code_words, self.sign_words = cw.value, ws.value

    def close(self):
        if getattr(self, "h", None):
            lib.tq_polar_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_kernel_path(self, path: int) -> None:
        _check(lib.tq_polar_set_kernel_path(self.h, path), "tq_polar_set_kernel_path")

    def alloc_codes(self, n: int, device="cuda") -> PolarCodes:
        codes = torch.zeros(n, self.code_words, dtype=torch.int32, device=device)
        r16 = torch.zeros(n, dtype=torch.int16, device=device)
        if not self.qjl:
            return PolarCodes(codes=codes, r16=r16)
        return PolarCodes(codes=codes, r16=r16, signs=torch.zeros(n, self.sign_words, dtype=torch.int32, device=device),
                          rnorm=torch.zeros(n, dtype=torch.int16, device=device))

    def quantize(self, x: torch.Tensor, out: PolarCodes | None = None, stream=None) -> PolarCodes:
        if x.dtype not in (torch.bfloat16, torch.float32):
            raise TypeError("x must be float32 or bfloat16")
        x2 = x.reshape(-1, self.d)
        if out is None:
            out = self.alloc_codes(x2.shape[0], device=x.device)
        dtype = TQ_BF16 if x.dtype == torch.bfloat16 else TQ_F32
        _check(lib.tq_polar_quantize(self.h, _ptr(x2), dtype, x2.shape[0], x2.stride(0), _ptr(out.codes),
                                     _ptr(out.r16), _ptr(out.signs), _ptr(out.rnorm), _stream(stream)),
               "tq_polar_quantize")
        return out

    def scores(self, q: torch.Tensor, keys: PolarCodes, scale: float = 1.0, out=None, stream=None) -> torch.Tensor:
        q2 = q.reshape(-1, self.d).contiguous().float()
        n = keys.codes.shape[0]
        if out is None:
            out = torch.empty(q2.shape[0], n, dtype=torch.float32, device=q.device)
        _check(lib.tq_polar_scores(self.h, _ptr(q2), q2.shape[0], _ptr(keys.codes), _ptr(keys.r16), _ptr(keys.signs),
                                   _ptr(keys.rnorm), n, scale, _ptr(out), _stream(stream)), "tq_polar_scores")
        return out

    def sync_status(self, stream=None) -> int:
        flags = _i(0)
        code = lib.tq_polar_sync_status(self.h, _stream(stream), ctypes.byref(flags))
        if code not in (TQ_OK, TQ_ERR_DEVICE):
            raise TQError(code, "tq_polar_sync_status")
        return flags.value


# ---------------------------------------------------------------------------------- paged decode step

@dataclass
class PagedCache:
    """Page pools of a compressed KV cache (layout of tq_paged_decode_step)."""
    kplanes: torch.Tensor
    ksigns: torch.Tensor
    knorm: torch.Tensor
    krnorm: torch.Tensor
    vplanes: torch.Tensor
    vnorm: torch.Tensor


def alloc_paged_cache(kctx: "Context", vctx: "Context", num_pages: int, Hkv: int, page_size: int,
                      device="cuda") -> PagedCache:
    lead = (num_pages, Hkv, page_size)
    return PagedCache(
        kplanes=torch.zeros(*lead, kctx.P, kctx.W, dtype=torch.int32, device=device),
        ksigns=torch.zeros(*lead, kctx.Ws, dtype=torch.int32, device=device),
        knorm=torch.zeros(*lead, dtype=torch.int16, device=device),
        krnorm=torch.zeros(*lead, dtype=torch.int16, device=device),
        vplanes=torch.zeros(*lead, vctx.P, vctx.W, dtype=torch.int32, device=device),
        vnorm=torch.zeros(*lead, dtype=torch.int16, device=device))


def paged_workspace(B, Hq, Hkv, max_pages, page_size, device="cuda") -> torch.Tensor:
    n = _sz()
    _check(lib.tq_paged_workspace_size(B, Hq, Hkv, max_pages, page_size, ctypes.byref(n)), "tq_paged_workspace_size")
    return torch.empty(n.value, dtype=torch.uint8, device=device)


def paged_decode_step(kctx: "Context", vctx: "Context", q, k_new, v_new, cache: PagedCache, block_table, length,
                      scale, out=None, workspace=None, stream=None):
    """One fused decode step (tq_paged_decode_step): appends k_new / v_new [B, Hkv, 128] at
    length[b], attends, advances length in place; returns out [B, Hq, 128]."""
    B, Hq, d = q.shape
    Hkv = k_new.shape[1]
    num_pages, _, page_size = cache.knorm.shape
    max_pages = block_table.shape[1]
    if k_new.dtype != v_new.dtype or k_new.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("k_new and v_new must both be float32 or bfloat16")
    dtype = TQ_BF16 if k_new.dtype == torch.bfloat16 else TQ_F32
    if out is None:
        out = torch.empty(B, Hq, d, device=q.device, dtype=torch.float32)
    if workspace is None:
        workspace = paged_workspace(B, Hq, Hkv, max_pages, page_size, device=q.device)
    kn, vn = k_new.contiguous(), v_new.contiguous()
    _check(lib.tq_paged_decode_step(kctx.h, vctx.h, _ptr(q.contiguous()), _ptr(kn), _ptr(vn), dtype, B, Hq, Hkv,
                                    _ptr(block_table), max_pages, page_size, num_pages, _ptr(length),
                                    _ptr(cache.kplanes), _ptr(cache.ksigns), _ptr(cache.knorm), _ptr(cache.krnorm),
                                    _ptr(cache.vplanes), _ptr(cache.vnorm), float(scale), _ptr(out), _ptr(workspace),
                                    workspace.numel(), _stream(stream)), "tq_paged_decode_step")
    return out
