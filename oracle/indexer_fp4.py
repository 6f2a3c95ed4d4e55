"""Oracle: indexer with FP4 query and key (a next hot-path row: no kernel yet).

Test infrastructure only (see ``oracle/__init__.py``).

What the pages fix
------------------
* The previous generation already trained the indexer's query and key for
  FP4 (quantization-aware training), and V4.1-Flash extends FP4 to the main
  KV cache ([P1] section 4, "Kuantisasi FP4 Main KV Cache").
* The main-KV FP4 format is E2M1 values with one E4M3 scale per 16 channels
  ([P3] section 3.2 "FP4 main KV"; [P1] sections 4 and 8).
* The indexer score is the weighted sum over heads of rectified head dot
  products, with blocks of 8 and the Full / Reindex selection of
  ``oracle.indexer`` ([P3] section 3.2 "Hierarchical Sparse Indexer").

Readings (the pages give no format for the indexer's FP4 values; each is
listed in the design notes):

* The indexer query (per head) and the indexer key (per position) use the
  main-KV format exactly: groups of 16 channels, scale = E4M3_rne_sat(amax/6),
  elements rounded to the nearest E2M1 level (``oracle.codec.quantize_rows``).
* The score is the exact indexer score of the dequantized values,
  ``s_t = sum_h w_h ReLU(dq(q_h) . dq(k_t))`` (``oracle.indexer.scores``):
  a dequantized value has at most 6 significant bits, so every product is
  exact in float64 and the head dots keep the exact-then-round-once rule.
* Storage: 64 bytes of codes + 8 bytes of scales = 72 bytes per key row of
  128 channels, against 128 bytes for E4M3 keys.
"""
from __future__ import annotations

import numpy as np

from . import codec, indexer

KEY_ROW_BYTES = 128 // 2 + 128 // codec.GROUP     # 64 B of codes + 8 B of scales


def quantize(x: np.ndarray):
    """Rows of bf16 / fp32 values (float64 [n, C], C a multiple of 32) to
    ``(codes uint8 [n, C/2], scales uint8 [n, C/16])`` in the main-KV format."""
    return codec.quantize_rows(np.asarray(x, dtype=np.float64))


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    return codec.dequantize_rows(codes, scales)


def scores(q_codes, q_scales, w, k_codes, k_scales) -> np.ndarray:
    """s_t = sum_h w_h ReLU(dq(q_h) . dq(k_t)) for every key row t (float64)."""
    return indexer.scores(dequantize(q_codes, q_scales), np.asarray(w, dtype=np.float64),
                          dequantize(k_codes, k_scales))


def full_topk(q, w, k, pool_blocks: int, topk: int):
    """Full mode with FP4 query and key: quantize both, then the Full-mode
    pool and Top-K of ``oracle.indexer`` over the dequantized values."""
    qc, qs = quantize(q)
    kc, ks = quantize(k)
    return indexer.full_topk(dequantize(qc, qs), np.asarray(w, dtype=np.float64),
                             dequantize(kc, ks), pool_blocks, topk)


def reindex_topk(q, w, k, pool, topk: int):
    """Reindex mode with FP4 query and key (the keys quantized as stored)."""
    qc, qs = quantize(q)
    kc, ks = quantize(k)
    return indexer.reindex_topk(dequantize(qc, qs), np.asarray(w, dtype=np.float64),
                                dequantize(kc, ks), pool, topk)
