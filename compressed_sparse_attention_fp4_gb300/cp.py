"""Context-parallel merge of the CSA2 decode path (one sequence over R ranks).

A 1M-position sequence can be split by context over R GPUs with one exchange
step (foosynaptic atlas "DeepSeek-V4.1-Flash 梗概", section 3.2,
"Hierarchical Sparse Indexer (decoder)": the Full layer scores every visible
position, keeps the Top-2048 blocks as the pool and the Top-K inside it;
Reindex layers score only the pool).  Rank r holds a contiguous, block-aligned
shard of the context and computes, on its shard only:

* Full layer: its local Top-P blocks, each with its exact block score (the
  max of its positions' scores); once the pool is merged, the local Top-K of
  the pool positions that fall in its shard, by their exact Full scores;
* Reindex layer: the same, with the Reindex layer's scores of those pool
  positions;
* attention: the partial (o_r, lse_r) over the selected entries of its shard
  (the rank holding the newest positions adds the SWA window).

All-gathers of (id, score) pairs (the pool, then the Top-K) and of the
(o, lse) partials, then the same rules as on one GPU, give the single-GPU
result exactly:

* selection: the global Top-k under (score desc, id asc) is the Top-k of the
  union of the local Top-k lists -- every globally selected item is among the
  k best of its own shard (for the pool: of the shard's blocks; for a Top-K:
  of the shard's pool positions);
* attention: a softmax over disjoint entry sets merges by log-sum-exp:
  M = max_r lse_r, o = sum_r e^(lse_r - M) o_r / sum_r e^(lse_r - M),
  lse = M + ln sum_r e^(lse_r - M).

This module holds the host-side merge and the collectives (torch.distributed,
any backend); the per-shard work would be the library's calls on each GPU's
shard.  It is exercised on CPU with gloo ranks; no multi-GPU run exists.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

BLOCK = 8


def shard_bounds(n_ctx: int, world: int, rank: int, block: int = BLOCK) -> tuple:
    """[lo, hi) positions of rank's contiguous shard; boundaries on blocks."""
    nb = -(-n_ctx // block)
    b0 = nb * rank // world
    b1 = nb * (rank + 1) // world
    return min(n_ctx, b0 * block), min(n_ctx, b1 * block)


def merge_selection(ids: torch.Tensor, scores: torch.Tensor, k: int) -> torch.Tensor:
    """Top-k of the union of R local lists under (score desc, id asc).

    ids: int64 [R, m] (-1 = empty slot); scores: float64 [R, m] (exact
    ranking values of the ids).  Returns int64 [k], ascending, -1 padded.
    """
    ids = ids.reshape(-1)
    scores = scores.reshape(-1).to(torch.float64)
    keep = ids >= 0
    ids, scores = ids[keep], scores[keep]
    # ascending id, then a stable descending sort by score: ties stay in id order
    o1 = torch.argsort(ids, stable=True)
    ids, scores = ids[o1], scores[o1]
    o2 = torch.argsort(scores, descending=True, stable=True)
    top = ids[o2][:k]
    out = torch.full((k,), -1, dtype=torch.int64, device=ids.device)
    out[:top.numel()] = torch.sort(top).values
    return out


def merge_attention(outs: torch.Tensor, lses: torch.Tensor) -> tuple:
    """Joint (o, lse) of R partials over disjoint entry sets.

    outs: [R, H, D]; lses: [R, H] (-inf for an empty partial, whose o is 0).
    Returns (o [H, D], lse [H]) in the inputs' floating type; an empty union
    gives o = 0 and lse = -inf.
    """
    m = torch.max(lses, dim=0).values                         # [H]
    finite = torch.isfinite(m)
    m_safe = torch.where(finite, m, torch.zeros_like(m))
    wts = torch.exp(lses - m_safe)                            # exp(-inf) = 0
    tot = wts.sum(dim=0)                                      # [H]
    num = (wts[:, :, None] * outs).sum(dim=0)                 # [H, D]
    nonempty = tot > 0
    o = torch.where(nonempty[:, None], num / torch.where(nonempty, tot, torch.ones_like(tot))[:, None],
                    torch.zeros_like(num))
    lse = torch.where(nonempty, m_safe + torch.log(torch.where(nonempty, tot, torch.ones_like(tot))),
                      torch.full_like(m, float("-inf")))
    return o, lse


def _all_gather(t: torch.Tensor, group=None) -> torch.Tensor:
    world = dist.get_world_size(group)
    parts = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(parts, t.contiguous(), group=group)
    return torch.stack(parts)


def gather_selection(local_ids: torch.Tensor, local_scores: torch.Tensor, k: int, group=None) -> torch.Tensor:
    """All-gather every rank's local Top-k (ids int64 [m], -1 padded; exact
    scores float64 [m]) and merge: the global Top-k, ascending, -1 padded."""
    return merge_selection(_all_gather(local_ids.to(torch.int64), group),
                           _all_gather(local_scores.to(torch.float64), group), k)


def gather_attention(out: torch.Tensor, lse: torch.Tensor, group=None) -> tuple:
    """All-gather every rank's attention partial (o [H, D], lse [H]) and merge."""
    return merge_attention(_all_gather(out, group), _all_gather(lse, group))
