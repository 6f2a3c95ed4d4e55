"""Host logic of the bench and the workloads (CPU only, no kernel runs).

* the algorithmic bytes the bench divides by: per indexer-key format (E4M3
  128 B, fp32 4 x Di, FP4 64 + 8 B per row) and per query count (q_len);
* the workloads' shapes: the FP4 and multi-query variants keep every other
  parameter of their base workload, and q_len = 1 draws exactly the values
  the single-query workloads always drew;
* the FP4 indexer-K buffer geometry the binding exposes (two planes).
"""
import numpy as np
import torch

import bench
from compressed_sparse_attention_fp4_gb300 import synth


def test_indexer_row_bytes_per_format():
    assert bench.idx_row_bytes(synth.workload("128k")) == 128
    assert bench.idx_row_bytes(synth.workload("tiny")) == 4 * 64
    assert bench.idx_row_bytes(synth.workload("1m-fp4")) == 64 + 8
    # the query stays bf16 for E4M3 and FP4 keys (16 heads x 128 x 2 B + 16 weights x 4 B)
    assert bench.idx_qw_bytes(synth.workload("128k")) == 16 * 128 * 2 + 64
    assert bench.idx_qw_bytes(synth.workload("1m-fp4")) == 16 * 128 * 2 + 64
    assert bench.idx_qw_bytes(synth.workload("tiny")) == 4 * 64 * 4 + 16


def test_scan_bytes_and_step_bytes():
    wl, w4 = synth.workload("1m"), synth.workload("1m-fp4")
    assert bench.kernel_bytes(wl, "indexer_scan_tc") == 128 * 1048576
    assert bench.kernel_bytes(w4, "indexer_scan_fp4") == 72 * 1048576
    assert bench.kernel_bytes(w4, "fp4_idx_quantize") == 2 * 128 + 72
    # FP4 keys: 56 B less per scanned position, plus the new key's write per Full layer
    d = bench.step_bytes(wl) - bench.step_bytes(w4)
    pool = 2048 * 8
    assert d == 56 * 1048576 + 56 * pool - (2 * 128 + 72)


def test_attention_bytes_scale_with_query_tokens():
    w1, w4 = synth.workload("128k"), synth.workload("128k-q4")
    a1, a4 = bench.attn_layer_bytes(w1), bench.attn_layer_bytes(w4)
    assert a1 == 512 * 416 + 128 * 1152 + 64 * 1152 + 64 * 513 * 4 + 512 * 4 == 567552
    assert a4 - a1 == 3 * 64 * (1152 + 513 * 4)
    assert bench.kernel_bytes(w4, "attn_cluster_tc") == 8 * a4


def test_workload_variants_keep_their_base():
    base, fp4, q4 = synth.workload("128k"), synth.workload("128k-fp4"), synth.workload("128k-q4")
    for v in (fp4, q4):
        assert v.ctx_lens == base.ctx_lens and v.schedule == base.schedule
        assert (v.heads, v.topk, v.swa, v.pool_blocks, v.idx_heads, v.idx_dim) == \
            (base.heads, base.topk, base.swa, base.pool_blocks, base.idx_heads, base.idx_dim)
    assert fp4.idx_k_dtype == "fp4" and fp4.q_len == 1
    assert q4.q_len == 4 and q4.idx_k_dtype == "fp8"
    assert synth.workload("1m-fp4").planted == synth.workload("1m").planted == 32


def test_query_draws():
    """q_len = 1 keeps the [H, 576] draw of the single-query workloads; q_len
    = 4 draws [4, H, 576] from the same stream (its first H rows are the
    single-query values)."""
    w1, w4 = synth.workload("tiny"), synth.workload("tiny", q_len=4)
    l1, l4 = synth.layer_inputs(w1, 0, 1), synth.layer_inputs(w4, 0, 1)
    assert l1["q"].shape == (16, 576) and l4["q"].shape == (4, 16, 576)
    np.testing.assert_array_equal(l4["q"][0], l1["q"])
    np.testing.assert_array_equal(l4["swa"], l1["swa"])
    # FP4 keys are drawn as bf16 rows (the library writes them as FP4)
    kv = synth.sequence_kv(synth.workload("1m-fp4"), 0, 0, 100)
    assert kv["idx_k"].dtype == np.uint16 and kv["idx_k"].shape == (100, 128)
    k8 = synth.sequence_kv(synth.workload("1m"), 0, 0, 100)["idx_k"]
    # the same normal draws: the E4M3 and bf16 roundings of one value share its sign bit
    f = (kv["idx_k"].astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_array_equal(np.signbit(f), (k8 & 0x80) != 0)


def test_fp4_indexer_k_planes():
    from compressed_sparse_attention_fp4_gb300 import csa2
    rows = 10
    buf = torch.arange(rows * 72, dtype=torch.int64).to(torch.uint8)
    codes, scales = csa2.fp4_idx_k_planes(buf, rows)
    assert codes.shape == (rows, 64) and scales.shape == (rows, 8)
    assert int(codes[3, 0]) == (3 * 64) % 256 and int(scales[2, 1]) == (rows * 64 + 2 * 8 + 1) % 256
