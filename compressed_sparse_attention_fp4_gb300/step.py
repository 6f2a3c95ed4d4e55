"""Decode-step runner: one query token per sequence through a CSA2 layer
schedule of Full / Reindex / Reuse layers, every step in libcsa2 kernels.

Layer modes (foosynaptic atlas "DeepSeek-V4.1-Flash 梗概", section 3.2, mode
table): Full runs the indexer over the whole context (new pool and Top-K),
Reindex re-scores the latest pool with its own indexer query (new Top-K),
Reuse keeps the latest Top-K; every layer then runs core attention with its
own query and SWA window.  Main KV and indexer K are one cache shared by all
layers.

The runner owns no method arithmetic: it orders the library calls, holds the
buffers between them and can capture the whole step in a CUDA graph.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import csa2


@dataclass
class StepBuffers:
    """Device tensors of one decode step (all on the same CUDA device)."""
    dims: csa2.Dims
    batch: int
    schedule: list
    # cache (shared by all layers)
    kv_codes: torch.Tensor          # uint8 [rows, 256]
    kv_scales: torch.Tensor         # uint8 [rows, 32]
    kv_rope: torch.Tensor           # bf16  [rows, 64]
    idx_k: torch.Tensor             # uint8 [rows, 128] (E4M3), fp32 [rows, 64] or uint8 [rows * 72] (FP4)
    page_table: torch.Tensor | None
    ctx_len: torch.Tensor           # int32 [B]
    # per-layer inputs
    q: torch.Tensor                 # bf16 [L, B, H, 576] ([L, B, q_len, H, 576] for q_len > 1)
    swa: torch.Tensor               # bf16 [L, B, W, 576]
    swa_len: torch.Tensor           # int32 [L, B]
    idx_q: torch.Tensor             # bf16 / fp32 [L, B, Hi, Di]
    idx_w: torch.Tensor             # fp32 [L, B, Hi]
    scale: float
    # optional decode-time append of the newest token at every Full layer
    new_latent: torch.Tensor | None = None   # bf16 [B, 512]
    new_rows: torch.Tensor | None = None     # int64 [B] cache rows of position N-1
    new_idx_k: torch.Tensor | None = None    # bf16 [B, 128]: its indexer key (FP4 indexer keys)
    idx_rows: int = 0                        # cache rows of the FP4 indexer-K buffer
    q_len: int = 1                           # query tokens per sequence (multi-query decode)
    # outputs
    out: torch.Tensor = None        # fp32 [L, B, (q_len,) H, 512]
    lse: torch.Tensor = None        # fp32 [L, B, (q_len,) H]
    topk: torch.Tensor = None       # int32 [L, B, K]  (indices each layer used)
    pool: torch.Tensor = None       # int32 [B, P]
    pool_len: torch.Tensor = None   # int32 [B]
    ws: torch.Tensor = None
    calls: int = 0                  # library calls of the last run_step

    def allocate_outputs(self):
        L, B, d = len(self.schedule), self.batch, self.dims
        dev = self.q.device
        qd = () if self.q_len == 1 else (self.q_len,)
        self.out = torch.empty((L, B) + qd + (d.heads, csa2.LATENT), dtype=torch.float32, device=dev)
        self.lse = torch.empty((L, B) + qd + (d.heads,), dtype=torch.float32, device=dev)
        self.topk = torch.full((L, B, d.topk), -1, dtype=torch.int32, device=dev)
        self.pool = torch.full((B, d.pool_blocks), -1, dtype=torch.int32, device=dev)
        self.pool_len = torch.zeros((B,), dtype=torch.int32, device=dev)
        self.ws = csa2.alloc_workspace(d, B, device=dev)
        return self


def step_calls(sb: StepBuffers, stream=None) -> list:
    """The library calls of one decode step, in order, as (label, thunk) pairs.

    Labels: ``append`` (FP4 write of the newest token's latent and, for FP4
    indexer keys, ``append_idx`` of its indexer key), ``F`` / ``Ri`` (the
    indexer of a Full / Reindex layer) and ``attn:<mode>`` (a layer's core
    attention), each with its layer number."""
    d, B = sb.dims, sb.batch
    if stream is None:
        stream = torch.cuda.current_stream()         # resolved once for the whole step
    calls = []
    cur = None
    for l, mode in enumerate(sb.schedule):
        if mode == "F":
            if sb.new_latent is not None and sb.new_idx_k is not None:
                calls.append((f"append_idx@{l}", lambda: csa2.fp4_idx_k_quantize_scatter(
                    sb.new_idx_k, sb.idx_k, sb.idx_rows, sb.new_rows, stream=stream)))
            # the keys are not written by the call before (an attention call, or
            # nothing) unless the newest token's FP4 key write precedes it
            fl = csa2.IDX_EARLY_INPUTS if sb.new_idx_k is None or sb.new_latent is None else 0
            calls.append((f"F@{l}", lambda l=l, fl=fl: csa2.indexer_full_topk(
                d, B, sb.idx_k, sb.page_table, sb.ctx_len, sb.idx_q[l], sb.idx_w[l], sb.pool,
                sb.pool_len, sb.topk[l], sb.ws, stream=stream, flags=fl)))
            if sb.new_latent is not None:
                # the newest token's latent goes into the main KV while the indexer
                # runs (the indexer reads no main-KV rows); attention comes after both
                calls.append((f"append@{l}", lambda: csa2.fp4_kv_quantize_scatter(
                    sb.new_latent, sb.new_rows, sb.kv_codes, sb.kv_scales, stream=stream,
                    flags=csa2.KV_EARLY_INPUTS)))
            cur = l
            m = csa2.MODE_FULL
        elif mode == "Ri":
            # follows an attention call, which writes none of the keys, lengths or pool
            calls.append((f"Ri@{l}", lambda l=l: csa2.indexer_reindex_topk(
                d, B, sb.idx_k, sb.page_table, sb.ctx_len, sb.idx_q[l], sb.idx_w[l], sb.pool,
                sb.pool_len, sb.topk[l], sb.ws, stream=stream, flags=csa2.IDX_EARLY_INPUTS)))
            cur = l
            m = csa2.MODE_REINDEX
        elif mode == "Ru":
            if cur is None:
                raise ValueError("a Reuse layer needs an earlier Full / Reindex layer")
            m = csa2.MODE_REUSE
        else:
            raise ValueError(f"unknown layer mode {mode!r}")
        if sb.q_len == 1:
            calls.append((f"attn:{mode}@{l}", lambda l=l, m=m, cur=cur: csa2.csa2_sparse_attn_decode(
                d, B, m, sb.q[l], sb.kv_codes, sb.kv_scales, sb.kv_rope, sb.page_table, sb.ctx_len,
                sb.topk[cur], sb.swa[l], sb.swa_len[l], sb.scale, sb.out[l], sb.lse[l], sb.ws,
                stream=stream)))
        else:
            calls.append((f"attn:{mode}@{l}", lambda l=l, m=m, cur=cur: csa2.csa2_sparse_attn_decode_mq(
                d, B, sb.q_len, m, sb.q[l], sb.kv_codes, sb.kv_scales, sb.kv_rope, sb.page_table,
                sb.ctx_len, sb.topk[cur], sb.swa[l], sb.swa_len[l], sb.scale, sb.out[l], sb.lse[l], sb.ws,
                stream=stream)))
    return calls


def run_step(sb: StepBuffers, stream=None, ncalls: int | None = None) -> int:
    """Enqueue one decode step (or its first `ncalls` library calls); returns
    the number of library calls made."""
    calls = step_calls(sb, stream)
    if ncalls is not None:
        calls = calls[:ncalls]
    for _, fn in calls:
        fn()
    sb.calls = len(calls)
    return len(calls)


class GraphedStep:
    """One decode step (or its first `ncalls` library calls) captured once in
    a CUDA graph and replayed."""

    def __init__(self, sb: StepBuffers, warmup: int = 1, ncalls: int | None = None):
        self.sb = sb
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(warmup):
                run_step(sb, ncalls=ncalls)
        torch.cuda.current_stream().wait_stream(s)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.calls = run_step(sb, ncalls=ncalls)

    def replay(self):
        self.graph.replay()
