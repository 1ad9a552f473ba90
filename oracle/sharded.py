"""The sequence- and database-sharded forms of the attention and search steps, plainly.

Test infrastructure only (see the package docstring for the citation legend).

The pages time attention logits over a compressed KV cache and top-k search over a coded
database on one GPU ([juejin §3]); they say nothing of several devices.  Reading taken for a
split across R processes (each holding a contiguous block of the sequence, or of the database
rows):

* attention: the softmax over the union of the blocks is assembled from one partial state per
  block and query head, (m, l, a) with m the block's largest logit, l = sum_i exp(logit_i - m)
  and a = sum_i exp(logit_i - m) v_i (an empty block: m = -inf, l = 0, a = 0).  With
  M = max_r m_r the output is  sum_r exp(m_r - M) a_r / sum_r exp(m_r - M) l_r,  which is the
  softmax-weighted sum of attention_values exactly (up to rounding).  For MSE-coded values
  a is kept in the value context's rotated basis (v_i = n16_i c[idx_i]) and the rotation back
  (Pi_v^T) is applied once after the merge, as attention_values' dequantisation would do
  per row (it is linear).
* search: every block returns its own top-k (global row numbers), and the global top-k is the
  top-k of the union of those lists under the same order (score descending, equal scores by
  row ascending): every row of the global top-k is in its own block's top-k.
"""

from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .codebook import Codebook
from .turboquant import Quantized, _group


def shard_bounds(n: int, world: int, rank: int) -> tuple[int, int]:
    """Rows [lo, hi) of block `rank` when n rows are cut into `world` contiguous blocks whose
    sizes differ by at most one."""
    return n * rank // world, n * (rank + 1) // world


def attention_partial(logits: np.ndarray, lens: np.ndarray, Hkv: int,
                      values_dense: Optional[np.ndarray] = None, values: Optional[Quantized] = None,
                      cb_v: Optional[Codebook] = None):
    """One block's partial states over its first lens[b] positions: m [B, Hq], l [B, Hq],
    a [B, Hq, d] (coded values: in the rotated basis, n16 c[idx])."""
    B, Hq, _ = logits.shape
    d = values_dense.shape[-1] if values_dense is not None else values.idx.shape[-1]
    m = np.full((B, Hq), -np.inf)
    l = np.zeros((B, Hq))
    a = np.zeros((B, Hq, d))
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        for h in range(Hq):
            g = _group(h, Hq, Hkv)
            x = np.asarray(logits[b, h, :L], dtype=np.float64)
            m[b, h] = np.max(x)
            e = np.exp(x - m[b, h])
            l[b, h] = np.sum(e)
            if values_dense is not None:
                V = np.asarray(values_dense[b, g, :L], dtype=np.float64)
            else:
                V = values.norm16[b, g, :L, None] * cb_v.centroids[values.idx[b, g, :L]]
            a[b, h] = e @ V
    return m, l, a


def merge_partials(parts: Sequence[tuple], Pi_v: Optional[np.ndarray] = None) -> np.ndarray:
    """Output [B, Hq, d] from the partial states (m, l, a) of R blocks; zeros where every block
    is empty.  Pi_v (coded values) rotates the merged sum back: o = Pi_v^T a (row form a @ Pi_v)."""
    M = np.max(np.stack([p[0] for p in parts]), axis=0)
    tot = np.zeros(M.shape)
    acc = np.zeros(parts[0][2].shape)
    for m, l, a in parts:
        w = np.where(np.isneginf(m), 0.0, np.exp(m - np.where(np.isneginf(M), 0.0, M)))
        tot += w * l
        acc += w[..., None] * a
    out = np.where(tot[..., None] > 0, acc / np.where(tot > 0, tot, 1.0)[..., None], 0.0)
    return out @ Pi_v if Pi_v is not None else out


def merge_topk(lists: Sequence[tuple], k: int) -> tuple[np.ndarray, np.ndarray]:
    """Global top-k [nq, k] from R blocks' (scores [nq, k_r], global rows [nq, k_r]) lists."""
    S = np.concatenate([np.asarray(s, dtype=np.float64) for s, _ in lists], axis=1)
    I = np.concatenate([np.asarray(i, dtype=np.int64) for _, i in lists], axis=1)
    k = min(k, S.shape[1])
    top_s = np.empty((S.shape[0], k))
    top_i = np.empty((S.shape[0], k), dtype=np.int64)
    for r in range(S.shape[0]):
        order = np.lexsort((I[r], -S[r]))[:k]
        top_s[r] = S[r, order]
        top_i[r] = I[r, order]
    return top_s, top_i
