"""Oracle for one fused decode step over a paged (block-table) KV cache.

TEST INFRASTRUCTURE (see the package docstring).  Plain float64 numpy; it reuses the pinned
contiguous functions (quantize, attention_output) after gathering the pages.

What the pages fix: the cache holds compressed keys and values and every decode step appends the
new token and scores all cached keys (juejin.cn post, section 三: attention logits over the KV
cache; csdn tutorial, section 背景: the cache of every token, the model's own replies included,
grows with the conversation).  Readings (the pages are silent on paging):

1. A page holds `page_size` consecutive token slots of one sequence for every KV head; the pools
   are [num_pages, Hkv, page_size, ...] and block_table[b][i] is the page of sequence b's tokens
   i * page_size .. (i + 1) * page_size - 1.
2. One step: quantize the new key (PROD mode) and value (MSE mode) of every (b, KV head), store
   them at position lens[b] (page block_table[b][lens[b] // page_size], slot lens[b] % page_size),
   then attend over positions 0 .. lens[b] (the new token included) and advance lens[b] by one.
"""
from __future__ import annotations

import numpy as np

from .turboquant import Quantized, attention_output, quantize


def alloc_pool(num_pages: int, Hkv: int, page_size: int, d: int, m: int = 0) -> Quantized:
    """Zeroed code pool [num_pages, Hkv, page_size, ...] (signs and rnorm16 when m > 0)."""
    z = Quantized(idx=np.zeros((num_pages, Hkv, page_size, d), dtype=np.int64),
                  norm16=np.zeros((num_pages, Hkv, page_size)))
    if m:
        z.signs = np.zeros((num_pages, Hkv, page_size, m), dtype=bool)
        z.rnorm16 = np.zeros((num_pages, Hkv, page_size))
    return z


def _put(pool: Quantized, page: int, h: int, slot: int, z: Quantized) -> None:
    pool.idx[page, h, slot] = z.idx[0]
    pool.norm16[page, h, slot] = z.norm16[0]
    if pool.signs is not None:
        pool.signs[page, h, slot] = z.signs[0]
        pool.rnorm16[page, h, slot] = z.rnorm16[0]


def gather(pool: Quantized, block_table: np.ndarray, lens: np.ndarray, page_size: int) -> Quantized:
    """Contiguous codes [B, Hkv, max(lens), ...] of each sequence's first lens[b] tokens."""
    B = len(lens)
    N = max(1, int(np.max(lens)))
    Hkv, d = pool.idx.shape[1], pool.idx.shape[3]
    out = Quantized(idx=np.zeros((B, Hkv, N, d), dtype=np.int64), norm16=np.zeros((B, Hkv, N)))
    if pool.signs is not None:
        out.signs = np.zeros((B, Hkv, N, pool.signs.shape[3]), dtype=bool)
        out.rnorm16 = np.zeros((B, Hkv, N))
    for b in range(B):
        for i in range(int(lens[b])):
            page, slot = int(block_table[b][i // page_size]), i % page_size
            out.idx[b, :, i] = pool.idx[page, :, slot]
            out.norm16[b, :, i] = pool.norm16[page, :, slot]
            if pool.signs is not None:
                out.signs[b, :, i] = pool.signs[page, :, slot]
                out.rnorm16[b, :, i] = pool.rnorm16[page, :, slot]
    return out


def paged_decode_step(q, k_new, v_new, kpool: Quantized, vpool: Quantized, block_table, lens, page_size: int,
                      Pi_k, S, cb_k, Pi_v, cb_v, scale: float):
    """Reading 2: append (in place, into the pools), attend, advance.  Returns (out [B, Hq, d],
    new lens)."""
    q = np.asarray(q, dtype=np.float64)
    lens = np.asarray(lens, dtype=np.int64)
    B, Hkv = k_new.shape[0], k_new.shape[1]
    for b in range(B):
        pos = int(lens[b])
        page, slot = int(block_table[b][pos // page_size]), pos % page_size
        for h in range(Hkv):
            _put(kpool, page, h, slot, quantize(np.asarray(k_new[b, h], dtype=np.float64)[None], Pi_k, cb_k, S))
            _put(vpool, page, h, slot, quantize(np.asarray(v_new[b, h], dtype=np.float64)[None], Pi_v, cb_v))
    new = lens + 1
    keys = gather(kpool, block_table, new, page_size)
    vals = gather(vpool, block_table, new, page_size)
    out = attention_output(q, keys, new, Pi_k, S, cb_k, scale, values=vals, Pi_v=Pi_v, cb_v=cb_v)
    return out, new
