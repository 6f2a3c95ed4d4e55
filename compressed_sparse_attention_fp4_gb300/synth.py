"""Seeded synthetic inputs for the CSA2 decode workloads.

This module only draws random numbers and stores them in the input formats
(bf16 bit patterns, E4M3 bytes, fp32).  It holds none of the method's
arithmetic (no quantization of the main KV, no scoring, no selection, no
attention); both the CUDA library's tests / benchmark and the CPU oracle
consume what it produces.

Every tensor is drawn from NumPy's PCG64 through ``SeedSequence`` children
keyed by (tensor, sequence, chunk), so any row range of any sequence can be
regenerated on its own, in any order, with the same values.

Workloads (shapes and value distributions of the decode configurations this
library targets):

``tiny``   B=1, N=4096, indexer K fp32 [N,64], 4 indexer heads, pool 64
           blocks, Top-128, 16 attention heads, SWA 128, schedule F,Ri,Ru.
``128k``   B=8, N=131,072, indexer K E4M3 [N,128], 16 indexer heads (bf16
           query), pool 2048 blocks, Top-512, 64 heads, SWA 128, schedule
           F, 5 x Reuse, Reindex, 5 x Reuse.
``1m``     B=1, N=1,048,576, as ``128k`` plus 32 planted positions drawn
           uniformly in [0, N/2) whose indexer-K row and latent are scaled by
           4 before rounding to the storage formats.
``1m-fp4`` / ``128k-fp4``  as ``1m`` / ``128k`` with FP4 indexer keys: the
           keys are drawn as bf16 rows and written to the cache by the
           library's FP4 indexer-key write (the query stays bf16).
``codec``  bf16 slab [1,048,576, 512], N(0,1), 5 outlier channels (1% of
           512, rounded) scaled by 20.
``128k-q4`` as ``128k`` with 4 query tokens per sequence and layer (the
           newest tokens, e.g. drafts a speculative step verifies): the
           attention query is [4, H, 576], the window and Top-K are shared.
``mix``    B=64, N_b uniform in [8192, 262144], KV in 64-position pages with
           a seeded random physical page order, schedule blocks of
           (F, Ru, Ru, Ri, Ru, Ru), as ``128k`` otherwise.

Value recipe: main-KV latent = N(0,1) x per-channel lognormal(0, 0.5) scale
(one scale vector per workload), rope part N(0,1), indexer K = N(0,1) x its
own per-channel lognormal(0, 0.5) scale, indexer query N(0,1), head weights
U(0,1), attention query N(0, sigma=1/sqrt(576)) (``q_sigma``), SWA rows drawn
like main-KV entries (latent channel scales on the first 512 channels).
Rounding to bf16 / E4M3 is round-to-nearest-even through PyTorch's CPU
conversions.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np
import torch

LATENT = 512
ROPE = 64
D_QK = LATENT + ROPE
PAGE = 64
CHUNK = 1 << 16          # rows per independently seeded chunk

# tensor ids for SeedSequence spawn keys
_T_LAT, _T_ROPE, _T_IDXK, _T_Q, _T_SWA, _T_IDXQ, _T_IDXW, _T_MISC = range(8)


@dataclass
class Workload:
    name: str
    ctx_lens: list
    idx_heads: int = 16
    idx_dim: int = 128
    idx_k_dtype: str = "fp8"            # "fp8" (E4M3), "fp32" or "fp4" (bf16 keys the library writes as FP4)
    heads: int = 64
    pool_blocks: int = 2048
    topk: int = 512
    swa: int = 128
    block: int = 8
    paged: bool = False
    schedule: list = field(default_factory=lambda: ["F"] + ["Ru"] * 5 + ["Ri"] + ["Ru"] * 5)
    q_sigma: float = 1.0 / math.sqrt(576.0)
    q_len: int = 1                      # query tokens per sequence and layer (multi-query decode)
    planted: int = 0
    planted_factor: float = 4.0
    seed: int = 0

    @property
    def batch(self) -> int:
        return len(self.ctx_lens)

    @property
    def max_ctx(self) -> int:
        return max(self.ctx_lens)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(float(D_QK))


def workload(name: str, **over) -> Workload:
    """The named decode workload (keyword overrides allowed for tests)."""
    sched_128k = ["F"] + ["Ru"] * 5 + ["Ri"] + ["Ru"] * 5
    if name == "tiny":
        wl = Workload("tiny", [4096], idx_heads=4, idx_dim=64, idx_k_dtype="fp32",
                      heads=16, pool_blocks=64, topk=128, schedule=["F", "Ri", "Ru"])
    elif name == "128k":
        wl = Workload("128k", [131072] * 8, schedule=sched_128k)
    elif name == "1m":
        wl = Workload("1m", [1048576], schedule=sched_128k, planted=32)
    elif name == "1m-fp4":
        wl = Workload("1m-fp4", [1048576], idx_k_dtype="fp4", schedule=sched_128k, planted=32)
    elif name == "128k-q4":
        wl = Workload("128k-q4", [131072] * 8, schedule=sched_128k, q_len=4)
    elif name == "128k-fp4":
        wl = Workload("128k-fp4", [131072] * 8, idx_k_dtype="fp4", schedule=sched_128k)
    elif name == "mix":
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(0, spawn_key=(_T_MISC, 1))))
        lens = rng.integers(8192, 262144, size=64, endpoint=True).tolist()
        wl = Workload("mix", lens, paged=True,
                      schedule=["F", "Ru", "Ru", "Ri", "Ru", "Ru"])
    else:
        raise KeyError(name)
    return replace(wl, **over) if over else wl


# --------------------------------------------------------------------------
# storage-format conversions (library rounding, no method arithmetic)
# --------------------------------------------------------------------------
def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 (RNE) bit patterns as uint16."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact widening)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    """float32 -> E4M3 (RNE) bytes; inputs are clamped to +-448 first."""
    x = np.clip(np.ascontiguousarray(x, dtype=np.float32), -448.0, 448.0)
    t = torch.from_numpy(x).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


# --------------------------------------------------------------------------
# random streams
# --------------------------------------------------------------------------
def _rng(wl: Workload, *key) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(wl.seed, spawn_key=key)))


def _chan_scale(wl: Workload, which: int, n: int) -> np.ndarray:
    return _rng(wl, _T_MISC, 10 + which).lognormal(0.0, 0.5, size=n).astype(np.float32)


def planted_positions(wl: Workload, b: int) -> np.ndarray:
    """Sorted planted positions of sequence b (empty if none)."""
    if not wl.planted:
        return np.zeros(0, dtype=np.int64)
    n = wl.ctx_lens[b]
    rng = _rng(wl, _T_MISC, 100, b)
    return np.sort(rng.choice(n // 2, size=wl.planted, replace=False)).astype(np.int64)


def _rows_chunks(lo: int, hi: int):
    c = lo // CHUNK
    while c * CHUNK < hi:
        a, z = max(lo, c * CHUNK), min(hi, (c + 1) * CHUNK)
        yield c, a, z
        c += 1


def _normal_rows(wl, tid, b, lo, hi, width):
    """N(0,1) float32 rows [lo, hi) of a (tensor, sequence) stream."""
    out = np.empty((hi - lo, width), dtype=np.float32)
    for c, a, z in _rows_chunks(lo, hi):
        rng = _rng(wl, tid, b, c)
        blk = rng.standard_normal((CHUNK, width), dtype=np.float32)
        out[a - lo:z - lo] = blk[a - c * CHUNK:z - c * CHUNK]
    return out


def sequence_kv(wl: Workload, b: int, lo: int = 0, hi: int | None = None):
    """Main-KV latent (bf16 bits), rope (bf16 bits) and indexer K rows [lo, hi).

    Returns dict ``latent`` uint16 [n, 512], ``rope`` uint16 [n, 64] and
    ``idx_k`` uint8 [n, Di] (E4M3), float32 [n, Di], or uint16 [n, Di]
    (bf16 bits, for the library's FP4 indexer-key write).
    """
    hi = wl.ctx_lens[b] if hi is None else hi
    lat = _normal_rows(wl, _T_LAT, b, lo, hi, LATENT) * _chan_scale(wl, 0, LATENT)
    rope = _normal_rows(wl, _T_ROPE, b, lo, hi, ROPE)
    ik = _normal_rows(wl, _T_IDXK, b, lo, hi, wl.idx_dim) * _chan_scale(wl, 1, wl.idx_dim)
    pl = planted_positions(wl, b)
    pl = pl[(pl >= lo) & (pl < hi)] - lo
    if pl.size:
        lat[pl] *= wl.planted_factor
        ik[pl] *= wl.planted_factor
    out = {"latent": to_bf16_bits(lat), "rope": to_bf16_bits(rope)}
    if wl.idx_k_dtype == "fp8":
        out["idx_k"] = to_e4m3_bytes(ik)
    elif wl.idx_k_dtype == "fp4":
        out["idx_k"] = to_bf16_bits(ik)
    else:
        out["idx_k"] = ik.astype(np.float32)
    return out


def sequence_kv_parallel(wl: Workload, b: int, threads: int | None = None):
    """``sequence_kv`` over the whole context, chunks generated in threads."""
    n = wl.ctx_lens[b]
    threads = threads or min(16, os.cpu_count() or 1)
    spans = [(a, min(n, a + CHUNK)) for a in range(0, n, CHUNK)]
    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(lambda s: sequence_kv(wl, b, s[0], s[1]), spans))
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}


def layer_inputs(wl: Workload, b: int, layer: int):
    """Per-layer inputs of sequence b: attention query, SWA rows, indexer q/w.

    ``q`` uint16 [H, 576] (bf16), ``swa`` uint16 [W, 576] (bf16),
    ``swa_len`` int, and for every layer (used only by Full / Reindex layers)
    ``idx_q`` [Hi, Di] (bf16 bits for the E4M3 and FP4 indexers, float32
    otherwise)
    and ``idx_w`` float32 [Hi].
    """
    r = _rng(wl, _T_Q, b, layer)
    q = r.standard_normal((wl.q_len * wl.heads, D_QK), dtype=np.float32) * np.float32(wl.q_sigma)
    q = q.reshape((wl.heads, D_QK) if wl.q_len == 1 else (wl.q_len, wl.heads, D_QK))
    r = _rng(wl, _T_SWA, b, layer)
    swa = r.standard_normal((wl.swa, D_QK), dtype=np.float32)
    swa[:, :LATENT] *= _chan_scale(wl, 0, LATENT)
    r = _rng(wl, _T_IDXQ, b, layer)
    iq = r.standard_normal((wl.idx_heads, wl.idx_dim), dtype=np.float32)
    r = _rng(wl, _T_IDXW, b, layer)
    iw = r.random(wl.idx_heads, dtype=np.float32)
    return {
        "q": to_bf16_bits(q),
        "swa": to_bf16_bits(swa),
        "swa_len": min(wl.swa, wl.ctx_lens[b]),
        "idx_q": to_bf16_bits(iq) if wl.idx_k_dtype in ("fp8", "fp4") else iq,
        "idx_w": iw,
    }


def page_table(wl: Workload):
    """Physical page order for a paged workload.

    Returns (table int32 [B, max_pages] with -1 padding, num_pages).  Pages of
    all sequences are numbered in sequence order and then shuffled by a
    seeded permutation.
    """
    pages = [-(-n // PAGE) for n in wl.ctx_lens]
    total = int(sum(pages))
    perm = _rng(wl, _T_MISC, 200).permutation(total).astype(np.int32)
    table = np.full((wl.batch, max(pages)), -1, dtype=np.int32)
    off = 0
    for b, p in enumerate(pages):
        table[b, :p] = perm[off:off + p]
        off += p
    return table, total


def codec_slab(n: int = 1 << 20, channels: int = LATENT, seed: int = 0,
               outliers: int | None = None, lo: int = 0, hi: int | None = None):
    """Rows [lo, hi) of the FP4 codec workload as bf16 bits [hi-lo, channels].

    N(0,1) values; ``outliers`` channels (default round(1% of channels)),
    picked by a seeded draw, are scaled by 20.
    """
    hi = n if hi is None else hi
    wl = Workload("codec", [n], seed=seed)
    k = int(round(0.01 * channels)) if outliers is None else outliers
    och = _rng(wl, _T_MISC, 300).choice(channels, size=k, replace=False)
    x = _normal_rows(wl, _T_LAT, 0, lo, hi, channels)
    x[:, och] *= 20.0
    return to_bf16_bits(x)
