"""Oracle: CSA2 decoder layer schedules (Full / Reindex / Reuse).

Test infrastructure only (see ``oracle/__init__.py``).

Every decoder layer has a static mode ([P3] section 3.2, mode table; [P2]
"CSA2: compressão em três dimensões"; [P4] section 3, "The Three Structural
Layers of CSA2"):

* Full    -- runs the indexer over every visible position: new candidate
             pool and new Top-K, then core attention.
* Reindex -- re-scores the latest Full layer's pool with its own indexer
             query: new Top-K, then core attention.
* Reuse   -- keeps the latest Top-K; only the attention query changes.

Reading: a Reuse layer uses the indices of the most recent Full or Reindex
layer, and a Reindex layer uses the pool (and indexer keys) of the most
recent Full layer.  Main KV and indexer K are one cache shared by all decoder
layers; each layer has its own SWA window and its own queries.

Schedules used by this library's workloads:

* ``tiny``  -- Full, Reindex, Reuse.
* ``128k``  -- Full, 5 x Reuse, Reindex, 5 x Reuse ("1 Full + 5 Reuse"
  blocks, [P2] same section).
* ``mix``   -- repeated blocks of (Full, Reuse, Reuse, Reindex, Reuse, Reuse):
  Full : Reindex : Reuse = 1 : 1 : 4.
"""
from __future__ import annotations

from . import attention, indexer

SCHEDULES = {
    "tiny": ["F", "Ri", "Ru"],
    "128k": ["F"] + ["Ru"] * 5 + ["Ri"] + ["Ru"] * 5,
    "mix": ["F", "Ru", "Ru", "Ri", "Ru", "Ru"],
}


def run_sequence(modes, idx_k, latent, rope, layers, pool_blocks, topk,
                 scale, block=indexer.BLOCK):
    """Run one sequence's decode token through a layer schedule.

    idx_k: [n_ctx, Di] indexer keys (float64); latent: [n_ctx, 512]
    dequantized main KV; rope: [n_ctx, 64].  ``layers[l]`` is a dict with
    ``q`` [H, 576], ``swa`` [W, 576], ``swa_len`` and, for Full / Reindex
    layers, ``idx_q`` [Hi, Di] and ``idx_w`` [Hi].
    Returns one dict per layer with ``mode``, ``topk``, ``out``, ``lse`` and,
    for Full layers, ``pool``; plus the indexer margins.
    """
    pool = None
    cur = None
    results = []
    for mode, lay in zip(modes, layers):
        rec = {"mode": mode}
        if mode == "F":
            r = indexer.full_topk(lay["idx_q"], lay["idx_w"], idx_k,
                                  pool_blocks, topk, block)
            pool, cur = r["pool"], r["topk"]
            rec.update(pool=pool, margin_pool=r["margin_pool"],
                       margin_topk=r["margin_topk"])
        elif mode == "Ri":
            if pool is None:
                raise ValueError("a Reindex layer needs an earlier Full layer")
            r = indexer.reindex_topk(lay["idx_q"], lay["idx_w"], idx_k, pool,
                                     topk, block)
            cur = r["topk"]
            rec.update(margin_topk=r["margin_topk"])
        elif mode == "Ru":
            if cur is None:
                raise ValueError("a Reuse layer needs an earlier Full/Reindex layer")
        else:
            raise ValueError(f"unknown layer mode {mode!r}")
        out, lse = attention.sparse_attn_decode(lay["q"], latent, rope, cur,
                                                lay["swa"], lay["swa_len"], scale)
        rec.update(topk=cur, out=out, lse=lse)
        results.append(rec)
    return results
