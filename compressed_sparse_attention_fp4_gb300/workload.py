"""Builds the device buffers of a synthetic decode workload.

Host data comes from ``synth`` (seeded draws in storage formats); the main-KV
cache is written by the library's own FP4 write path (``fp4_kv_quantize`` /
``fp4_kv_quantize_scatter``), exactly as a serving engine would fill it.
Indexer K, rope and the per-layer inputs are copied as drawn, except FP4
indexer keys, which the library's FP4 indexer-key write stores.
"""
from __future__ import annotations

import numpy as np
import torch

from . import csa2, synth
from .step import StepBuffers


_IDXK = {"fp8": csa2.IDXK_E4M3, "fp32": csa2.IDXK_F32, "fp4": csa2.IDXK_FP4}


def dims_for(wl: synth.Workload) -> csa2.Dims:
    d = csa2.Dims(idx_heads=wl.idx_heads, idx_dim=wl.idx_dim, idx_k_dtype=_IDXK[wl.idx_k_dtype],
                  pool_blocks=wl.pool_blocks, topk=wl.topk, heads=wl.heads, swa=wl.swa,
                  max_ctx=wl.max_ctx)
    if wl.paged:
        table, total = synth.page_table(wl)
        d.max_pages = table.shape[1]
        d.num_pages = total
        d.max_ctx = table.shape[1] * csa2.PAGE
    return d


def _u16(t: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(t).view(np.int16))


def cache_rows(wl: synth.Workload, b: int, n: int, table) -> np.ndarray:
    """Physical cache rows of positions [0, n) of sequence b."""
    t = np.arange(n, dtype=np.int64)
    if table is None:
        return b * wl.max_ctx + t
    return table[b, t // csa2.PAGE].astype(np.int64) * csa2.PAGE + t % csa2.PAGE


def build(wl: synth.Workload, device="cuda", threads=None, keep_new_token=True) -> StepBuffers:
    """Upload a workload and return ready-to-run step buffers."""
    dims = dims_for(wl)
    B = wl.batch
    dev = torch.device(device)
    table = None
    if wl.paged:
        table, total = synth.page_table(wl)
        rows = total * csa2.PAGE
    else:
        rows = B * wl.max_ctx
    codes = torch.zeros((rows, 256), dtype=torch.uint8, device=dev)
    scales = torch.zeros((rows, 32), dtype=torch.uint8, device=dev)
    rope = torch.zeros((rows, 64), dtype=torch.bfloat16, device=dev)
    fp4k = wl.idx_k_dtype == "fp4"
    if wl.idx_k_dtype == "fp8":
        idx_k = torch.zeros((rows, wl.idx_dim), dtype=torch.uint8, device=dev)
    elif fp4k:
        idx_k = torch.zeros((rows * 72,), dtype=torch.uint8, device=dev)   # codes [rows][64], scales [rows][8]
        new_idx_k = torch.zeros((B, wl.idx_dim), dtype=torch.bfloat16, device=dev)
    else:
        idx_k = torch.zeros((rows, wl.idx_dim), dtype=torch.float32, device=dev)
    new_latent = torch.zeros((B, 512), dtype=torch.bfloat16, device=dev)
    new_rows = torch.zeros((B,), dtype=torch.int64, device=dev)
    for b in range(B):
        n = wl.ctx_lens[b]
        kv = synth.sequence_kv_parallel(wl, b, threads)
        dst = torch.from_numpy(cache_rows(wl, b, n, table)).to(dev)
        lat = _u16(kv["latent"]).to(dev).view(torch.bfloat16)
        csa2.fp4_kv_quantize_scatter(lat, dst, codes, scales)
        rope.index_copy_(0, dst, _u16(kv["rope"]).to(dev).view(torch.bfloat16))
        if fp4k:
            ik = _u16(kv["idx_k"]).to(dev).view(torch.bfloat16)
            csa2.fp4_idx_k_quantize_scatter(ik, idx_k, rows, dst)
            new_idx_k[b] = ik[n - 1]
        else:
            ik = torch.from_numpy(np.ascontiguousarray(kv["idx_k"])).to(dev)
            idx_k.index_copy_(0, dst, ik)
        new_latent[b] = lat[n - 1]
        new_rows[b] = dst[n - 1]
        del lat
    L = len(wl.schedule)
    H, W, Hi, Di = wl.heads, wl.swa, wl.idx_heads, wl.idx_dim
    qshape = (L, B, H, synth.D_QK) if wl.q_len == 1 else (L, B, wl.q_len, H, synth.D_QK)
    q = np.empty(qshape, dtype=np.uint16)
    swa = np.empty((L, B, W, synth.D_QK), dtype=np.uint16)
    swa_len = np.empty((L, B), dtype=np.int32)
    bf16_q = wl.idx_k_dtype in ("fp8", "fp4")
    iq = np.empty((L, B, Hi, Di), dtype=np.uint16 if bf16_q else np.float32)
    iw = np.empty((L, B, Hi), dtype=np.float32)
    for l in range(L):
        for b in range(B):
            li = synth.layer_inputs(wl, b, l)
            q[l, b], swa[l, b], swa_len[l, b] = li["q"], li["swa"], li["swa_len"]
            iq[l, b], iw[l, b] = li["idx_q"], li["idx_w"]
    iq_t = _u16(iq).view(torch.bfloat16) if bf16_q else torch.from_numpy(iq)
    sb = StepBuffers(
        dims=dims, batch=B, schedule=list(wl.schedule),
        kv_codes=codes, kv_scales=scales, kv_rope=rope, idx_k=idx_k,
        page_table=None if table is None else torch.from_numpy(table).to(dev),
        ctx_len=torch.tensor(wl.ctx_lens, dtype=torch.int32, device=dev),
        q=_u16(q).view(torch.bfloat16).to(dev), swa=_u16(swa).view(torch.bfloat16).to(dev),
        swa_len=torch.from_numpy(swa_len).to(dev), idx_q=iq_t.to(dev),
        idx_w=torch.from_numpy(iw).to(dev), scale=wl.scale,
        new_latent=new_latent if keep_new_token else None,
        new_rows=new_rows if keep_new_token else None,
        new_idx_k=new_idx_k if (fp4k and keep_new_token) else None, idx_rows=rows, q_len=wl.q_len)
    return sb.allocate_outputs()
