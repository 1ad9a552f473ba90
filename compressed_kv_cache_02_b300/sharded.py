"""Attention and search over blocks held by several processes, one GPU each.

Each process holds one contiguous block of every cached sequence (positions [lo, hi) of the
KV cache, `shard_bounds`), or one block of the database rows.  The pages time both operations on
one GPU (juejin.cn post, section 三); cutting them across processes is exact:

* attention logits are local (the query is replicated to every process);
* the softmax and the value sum need one exchange: every process computes its block's partial
  state per (batch, query head), (max logit, sum of weights, weighted value sum), with
  tq_attn_values_partial; the states are all-gathered; every process merges them by their maxima
  (log-sum-exp) and rotates back once (tq_attn_merge_partials);
* search: every process returns its block's top-k with tq_search_topk, the lists are
  all-gathered, and tq_topk_merge keeps the k best under the same order (score descending, equal
  scores by global row ascending), which is the unsharded result since every row of the global
  top-k is in its own block's top-k.

The exchange is torch.distributed's all-gather on the process group (NCCL between GPUs; on a gloo
group the tensors travel through host memory).  The device work goes through `ops` (default: the
library's calls, `TqOps`); a caller may pass another object with the same methods.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

INT32_MAX = 2 ** 31 - 1


def shard_bounds(n: int, world: int, rank: int) -> tuple[int, int]:
    """Rows [lo, hi) of block `rank` when n rows are cut into `world` contiguous blocks whose sizes
    differ by at most one."""
    return n * rank // world, n * (rank + 1) // world


def block_lengths(length: torch.Tensor, lo: int, hi: int) -> torch.Tensor:
    """Positions of each sequence (global lengths `length` [B]) that fall in the block [lo, hi)."""
    return (length.to(torch.int64) - lo).clamp(0, hi - lo).to(torch.int32)


class TqOps:
    """The library's calls on the current GPU (libtq through its binding)."""

    score_dtype = torch.float32   # of the scores search_topk returns

    @staticmethod
    def _tq():
        from . import tq
        return tq

    def rows(self, db) -> int:
        return int(db.planes.shape[0])

    def logits(self, kctx, q, keys, cap, length, scale):
        return kctx.attn_logits(q, keys, cap, length, scale)

    def values_partial(self, logits, length, values, vctx):
        return self._tq().attn_values_partial(logits, length, values, vctx=vctx)

    def merge_partials(self, parts, vctx):
        return self._tq().attn_merge_partials(parts, vctx=vctx)

    def search_topk(self, ctx, q, db, k):
        return ctx.search_topk(q, db, k)

    def topk_merge(self, cand_s, cand_i, row_offsets):
        return self._tq().topk_merge(cand_s, cand_i, row_offsets)


def all_gather(t: torch.Tensor, group=None) -> torch.Tensor:
    """[world, *t.shape]: every process's t, in rank order."""
    world = dist.get_world_size(group)
    via_host = t.is_cuda and dist.get_backend(group) == "gloo"
    src = (t.cpu() if via_host else t).contiguous()
    parts = [torch.empty_like(src) for _ in range(world)]
    dist.all_gather(parts, src, group=group)
    out = torch.stack(parts)
    return out.to(t.device) if via_host else out


def attention_values(logits, length, values, vctx=None, group=None, ops=None):
    """Softmax over every block's logits and the weighted sum of every block's values; each process
    gets the whole output [B, Hq, d].  logits [B, Hq, cap_r] and values (bf16 [B, Hkv, cap_r, d],
    or the Codes of an MSE-mode vctx) are this process's block; length [B] (device int32) the
    number of positions of each sequence the block holds (`block_lengths`)."""
    ops = ops or TqOps()
    part = ops.values_partial(logits, length, values, vctx)
    return ops.merge_partials(all_gather(part, group), vctx)


def decode_attention(kctx, q, keys, cap, length, scale, values, vctx=None, group=None, ops=None):
    """One decode step's attention over a sequence-sharded compressed cache: the logits of the
    block (local), then `attention_values` (one all-gather)."""
    ops = ops or TqOps()
    logits = ops.logits(kctx, q, keys, cap, length, scale)
    return attention_values(logits, length, values, vctx, group, ops)


def search_topk(ctx, q, db, k, row_offset, group=None, ops=None):
    """Global top-k (scores, global rows) [nq, k] over every process's database block; db holds this
    process's rows, the first of them global row `row_offset`.  A block with fewer than k rows
    contributes all of them."""
    ops = ops or TqOps()
    n = ops.rows(db)
    kk = min(k, n)
    nq = q.shape[0]
    s = torch.full((nq, k), float("-inf"), dtype=ops.score_dtype, device=q.device)
    i = torch.full((nq, k), INT32_MAX, dtype=torch.int32, device=q.device)
    if kk > 0:
        bs, bi = ops.search_topk(ctx, q, db, kk)
        s[:, :kk] = bs.to(s.dtype)
        i[:, :kk] = bi.to(i.dtype)
    offs = all_gather(torch.tensor([row_offset], dtype=torch.int64, device=q.device), group)
    return ops.topk_merge(all_gather(s, group), all_gather(i, group), offs.reshape(-1).cpu().tolist())
