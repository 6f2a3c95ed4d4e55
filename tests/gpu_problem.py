"""Small, hand-shaped device problems for the GPU parity tests.

Draws seeded inputs (no method arithmetic) and lays them out on the device in
the library's cache format; the oracle side gets the same values widened to
float64.
"""
import numpy as np
import torch

from compressed_sparse_attention_fp4_gb300 import csa2, synth
from tests.helpers import bf16_f64, idxk_f64


class Problem:
    pass


def make_problem(ctx_lens, Hi=16, Di=128, dtype="fp8", P=2048, K=512, H=64, W=128,
                 paged=False, seed=0, kind="random", q_sigma=None, with_kv=True):
    rng = np.random.default_rng(seed)
    p = Problem()
    p.ctx_lens = list(ctx_lens)
    B = len(ctx_lens)
    p.B, p.Hi, p.Di, p.dtype, p.P, p.K, p.H, p.W = B, Hi, Di, dtype, P, K, H, W
    max_ctx = max(max(ctx_lens), 1)
    if paged:
        pages = [-(-n // 64) for n in ctx_lens]
        total = sum(pages) + 3                         # a few unused pages
        perm = rng.permutation(total).astype(np.int32)
        table = np.full((B, max(max(pages), 1)), -1, dtype=np.int32)
        off = 0
        for b, pg in enumerate(pages):
            table[b, :pg] = perm[off:off + pg]
            off += pg
        p.table = table
        rows = total * 64
        dims = csa2.Dims(idx_heads=Hi, idx_dim=Di,
                         idx_k_dtype=csa2.IDXK_E4M3 if dtype == "fp8" else csa2.IDXK_F32,
                         pool_blocks=P, topk=K, heads=H, swa=W, max_pages=table.shape[1],
                         num_pages=total, max_ctx=table.shape[1] * 64)
    else:
        p.table = None
        rows = B * max_ctx
        dims = csa2.Dims(idx_heads=Hi, idx_dim=Di,
                         idx_k_dtype=csa2.IDXK_E4M3 if dtype == "fp8" else csa2.IDXK_F32,
                         pool_blocks=P, topk=K, heads=H, swa=W, max_ctx=max_ctx)
    p.dims = dims
    p.rows_of = []
    for b, n in enumerate(ctx_lens):
        t = np.arange(n, dtype=np.int64)
        if paged:
            p.rows_of.append(table[b, t // 64].astype(np.int64) * 64 + t % 64)
        else:
            p.rows_of.append(b * max_ctx + t)
    # indexer keys
    scale_ch = rng.lognormal(0, 0.5, Di).astype(np.float32)
    p.idx_k_raw = []
    if dtype == "fp8":
        dev_k = np.zeros((rows, Di), dtype=np.uint8)
    else:
        dev_k = np.zeros((rows, Di), dtype=np.float32)
    for b, n in enumerate(ctx_lens):
        if kind in ("trunc", "cancel"):
            # E4M3 codes built directly: channel 0 (and 1) at 448, the rest small
            # positive values just below a power of two (worst case for products
            # truncated against the largest one of an MMA step)
            raw = ((rng.integers(1, 6, (n, Di)) << 3) | 7).astype(np.uint8)
            raw[:, 0] = 0x7E
            if kind == "cancel":
                raw[:, 1] = 0x7E
            raw[:, 32::32] = 0x7E                      # one large product in every K step
            p.idx_k_raw.append(raw)
            dev_k[p.rows_of[b]] = raw
            continue
        if kind in ("ties", "wide"):
            base = rng.standard_normal((3, Di)).astype(np.float32) * scale_ch
            if kind == "wide":
                # (fp32 keys) products spanning more than 126 bits: channel 0
                # large, channels 1-3 near the bottom of the fp32 normal range
                base[:, 0] *= np.float32(2.0 ** 12)
                base[:, 1:4] *= np.float32(2.0 ** -100)
            k = base[rng.integers(0, 3, n)]
        else:
            k = rng.standard_normal((n, Di)).astype(np.float32) * scale_ch
        raw = synth.to_e4m3_bytes(k) if dtype == "fp8" else k.astype(np.float32)
        p.idx_k_raw.append(raw)
        dev_k[p.rows_of[b]] = raw
    p.idx_k = torch.from_numpy(dev_k).cuda()
    q = rng.standard_normal((B, Hi, Di)).astype(np.float32)
    if kind in ("trunc", "cancel"):
        q = np.abs(q) * np.float32(2.0 ** -7)
        q[:, :, 0] = 1.0
        q[:, :, 32::32] = 1.0
        if kind == "cancel":
            q[:, :, 1] = -1.0                          # k0 q0 + k1 q1 = 0 exactly
    p.idx_q_raw = synth.to_bf16_bits(q) if dtype == "fp8" else q
    p.idx_q_f64 = bf16_f64(p.idx_q_raw) if dtype == "fp8" else q.astype(np.float64)
    p.idx_q = (torch.from_numpy(p.idx_q_raw.view(np.int16)).view(torch.bfloat16)
               if dtype == "fp8" else torch.from_numpy(q)).cuda()
    p.w_raw = rng.random((B, Hi)).astype(np.float32)
    p.w = torch.from_numpy(p.w_raw).cuda()
    p.ctx = torch.tensor(ctx_lens, dtype=torch.int32, device="cuda")
    p.page_table = None if p.table is None else torch.from_numpy(p.table).cuda()
    if with_kv:
        lat_scale = rng.lognormal(0, 0.5, 512).astype(np.float32)
        p.latent_raw, p.rope_raw = [], []
        codes = torch.zeros((rows, 256), dtype=torch.uint8, device="cuda")
        scales = torch.zeros((rows, 32), dtype=torch.uint8, device="cuda")
        rope = torch.zeros((rows, 64), dtype=torch.bfloat16, device="cuda")
        for b, n in enumerate(ctx_lens):
            lat = synth.to_bf16_bits(rng.standard_normal((n, 512)).astype(np.float32) * lat_scale)
            rp = synth.to_bf16_bits(rng.standard_normal((n, 64)).astype(np.float32))
            p.latent_raw.append(lat)
            p.rope_raw.append(rp)
            if n:
                dst = torch.from_numpy(p.rows_of[b]).cuda()
                x = torch.from_numpy(lat.view(np.int16)).cuda().view(torch.bfloat16)
                csa2.fp4_kv_quantize_scatter(x, dst, codes, scales)
                rope.index_copy_(0, dst, torch.from_numpy(rp.view(np.int16)).cuda().view(torch.bfloat16))
        p.codes, p.scales, p.rope = codes, scales, rope
        sig = (1.0 / np.sqrt(576.0)) if q_sigma is None else q_sigma
        qa = rng.standard_normal((B, H, 576)).astype(np.float32) * sig
        p.q_raw = synth.to_bf16_bits(qa)
        p.q = torch.from_numpy(p.q_raw.view(np.int16)).cuda().view(torch.bfloat16)
        swa = rng.standard_normal((B, max(W, 1), 576)).astype(np.float32)
        p.swa_raw = synth.to_bf16_bits(swa)
        p.swa = torch.from_numpy(p.swa_raw.view(np.int16)).cuda().view(torch.bfloat16)
        p.swa_len_np = np.array([min(W, n) for n in ctx_lens], dtype=np.int32)
        p.swa_len = torch.from_numpy(p.swa_len_np).cuda()
    p.ws = csa2.alloc_workspace(dims, B)
    return p


def oracle_keys(p, b):
    return idxk_f64(p.idx_k_raw[b], p.dtype)


def run_full(p):
    pool = torch.full((p.B, p.P), -7, dtype=torch.int32, device="cuda")
    plen = torch.zeros((p.B,), dtype=torch.int32, device="cuda")
    topk = torch.full((p.B, p.K), -7, dtype=torch.int32, device="cuda")
    csa2.indexer_full_topk(p.dims, p.B, p.idx_k, p.page_table, p.ctx, p.idx_q, p.w, pool, plen,
                           topk, p.ws)
    torch.cuda.synchronize()
    return pool, plen, topk


def run_reindex(p, pool, plen, q=None, w=None):
    topk = torch.full((p.B, p.K), -7, dtype=torch.int32, device="cuda")
    csa2.indexer_reindex_topk(p.dims, p.B, p.idx_k, p.page_table, p.ctx,
                              p.idx_q if q is None else q, p.w if w is None else w,
                              pool, plen, topk, p.ws)
    torch.cuda.synchronize()
    return topk


def make_fp4_problem(ctx_lens, Hi=16, P=2048, K=512, paged=False, seed=0, kind="random"):
    """Indexer-only problem with FP4 keys: bf16 keys are drawn, written into the
    two-plane FP4 indexer-K buffer by the library's quantize call, and kept as
    float64 for the oracle (which quantizes them itself)."""
    rng = np.random.default_rng(seed)
    p = Problem()
    p.ctx_lens = list(ctx_lens)
    B = len(ctx_lens)
    p.B, p.Hi, p.Di, p.P, p.K = B, Hi, 128, P, K
    max_ctx = max(max(ctx_lens), 1)
    if paged:
        pages = [-(-n // 64) for n in ctx_lens]
        total = sum(pages) + 3
        perm = rng.permutation(total).astype(np.int32)
        table = np.full((B, max(max(pages), 1)), -1, dtype=np.int32)
        off = 0
        for b, pg in enumerate(pages):
            table[b, :pg] = perm[off:off + pg]
            off += pg
        p.table = table
        rows = total * 64
        dims = csa2.Dims(idx_heads=Hi, idx_dim=128, idx_k_dtype=csa2.IDXK_FP4, pool_blocks=P, topk=K,
                         heads=64, swa=128, max_pages=table.shape[1], num_pages=total,
                         max_ctx=table.shape[1] * 64)
    else:
        p.table = None
        rows = B * max_ctx
        dims = csa2.Dims(idx_heads=Hi, idx_dim=128, idx_k_dtype=csa2.IDXK_FP4, pool_blocks=P, topk=K,
                         heads=64, swa=128, max_ctx=max_ctx)
    p.dims, p.rows = dims, rows
    p.rows_of = []
    for b, n in enumerate(ctx_lens):
        t = np.arange(n, dtype=np.int64)
        p.rows_of.append(table[b, t // 64].astype(np.int64) * 64 + t % 64 if paged else b * max_ctx + t)
    scale_ch = rng.lognormal(0, 0.5, 128).astype(np.float32)
    p.k_bits = []
    p.idx_k = torch.zeros(rows * 72, dtype=torch.uint8, device="cuda")
    for b, n in enumerate(ctx_lens):
        if kind == "ties":
            base = rng.standard_normal((3, 128)).astype(np.float32) * scale_ch
            k = base[rng.integers(0, 3, n)]
        elif kind == "wide":
            # every group of 16 at its own power-of-two scale across the E4M3
            # range: group terms of very different size, with cancellation
            k = rng.standard_normal((n, 128)).astype(np.float32)
            k *= np.repeat(np.exp2(rng.integers(-8, 8, (n, 8))), 16, axis=1).astype(np.float32)
        else:
            k = rng.standard_normal((n, 128)).astype(np.float32) * scale_ch
        bits = synth.to_bf16_bits(k)
        p.k_bits.append(bits)
        if n:
            x = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
            csa2.fp4_idx_k_quantize_scatter(x, p.idx_k, rows, torch.from_numpy(p.rows_of[b]).cuda())
    q = rng.standard_normal((B, Hi, 128)).astype(np.float32)
    if kind == "wide":
        q *= np.repeat(np.exp2(rng.integers(-6, 6, (B, Hi, 8))), 16, axis=2).astype(np.float32)
    p.idx_q_raw = synth.to_bf16_bits(q)
    p.idx_q_f64 = bf16_f64(p.idx_q_raw)
    p.idx_q = torch.from_numpy(p.idx_q_raw.view(np.int16)).view(torch.bfloat16).cuda()
    p.w_raw = rng.random((B, Hi)).astype(np.float32)
    p.w = torch.from_numpy(p.w_raw).cuda()
    p.ctx = torch.tensor(ctx_lens, dtype=torch.int32, device="cuda")
    p.page_table = None if p.table is None else torch.from_numpy(p.table).cuda()
    p.ws = csa2.alloc_workspace(dims, B)
    return p


def fp4_keys_f64(p, b):
    """The bf16 keys of sequence b as float64 (before quantization)."""
    return bf16_f64(p.k_bits[b])
