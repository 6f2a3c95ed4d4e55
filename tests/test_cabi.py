"""The C-ABI library loads on a CPU host, exports every function that
include/csa2.h declares, and rejects bad arguments on the host (before any
CUDA call, so these run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def mod():
    from compressed_sparse_attention_fp4_gb300 import build
    build.build()
    from compressed_sparse_attention_fp4_gb300 import csa2
    return csa2


def test_header_functions_exported(mod):
    names = declared_functions()
    assert len(names) >= 11
    lib = ctypes.CDLL(mod.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(mod.SIGNATURES), set(names) - set(mod.SIGNATURES)


def test_version_and_strings(mod):
    assert mod.version() == 100
    for code, name in mod.STATUS.items():
        assert mod._lib.csa2_status_string(code).decode() == name


def test_workspace_size_and_shape_checks(mod):
    d = mod.Dims(max_ctx=131072)
    assert mod.workspace_size(d, 8) > 8 * 131072 * 4
    bad = [dict(idx_heads=17), dict(idx_heads=0), dict(idx_dim=64), dict(pool_blocks=4096),
           dict(topk=4096), dict(heads=128), dict(swa=256), dict(max_ctx=(1 << 20) + 1)]
    for kw in bad:
        with pytest.raises(mod.Csa2Error) as e:
            mod.workspace_size(mod.Dims(**{**d.__dict__, **kw}), 1)
        assert e.value.code == 2, kw
    with pytest.raises(mod.Csa2Error) as e:
        mod.workspace_size(mod.Dims(idx_k_dtype=7), 1)
    assert e.value.code == 1
    with pytest.raises(mod.Csa2Error):
        mod.workspace_size(d, -1)


def test_host_argument_errors(mod):
    lib = mod._lib
    d = mod.Dims(max_ctx=1024, pool_blocks=64, topk=128)
    dc = ctypes.byref(d.c())
    P = ctypes.c_void_p
    fake = P(0x10000)           # never dereferenced: validation fails first
    assert lib.fp4_kv_quantize(None, 5, fake, fake, None) == 1
    assert lib.fp4_kv_quantize(fake, -1, fake, fake, None) == 1
    assert lib.fp4_kv_quantize(P(0x10001), 5, fake, fake, None) == 1      # misaligned
    assert lib.fp4_kv_quantize(None, 0, None, None, None) == 0            # empty: no-op
    assert lib.fp4_kv_dequantize(fake, None, 3, fake, None) == 1
    assert lib.fp4_kv_quantize_scatter(fake, 2, None, fake, fake, None) == 1
    ws = mod.workspace_size(d, 2)
    # workspace too small / misaligned / missing
    args = [fake, None] + [fake] * 6          # contiguous cache: no page table
    assert lib.indexer_full_topk(dc, 2, *args, fake, ws - 1, None) == 3
    assert lib.indexer_full_topk(dc, 2, *args, P(0x10010), ws, None) == 1
    assert lib.indexer_full_topk(dc, 2, *args, None, ws, None) == 1
    # null input with a big-enough workspace
    assert lib.indexer_full_topk(dc, 2, None, *args[1:], fake, ws, None) == 1
    assert lib.indexer_reindex_topk(dc, 2, fake, None, *([fake] * 4), None, fake, fake, ws, None) == 1
    # attention: bad mode, null swa with a window, NaN scale
    a = [fake] * 4 + [None] + [fake] * 4      # no page table
    assert lib.csa2_sparse_attn_decode(dc, 2, 3, *a, 0.1, fake, fake, fake, ws, None) == 1
    assert lib.csa2_sparse_attn_decode(dc, 2, 0, *a[:7], None, fake, 0.1, fake, fake, fake, ws, None) == 1
    assert lib.csa2_sparse_attn_decode(dc, 2, 0, *a, float("nan"), fake, fake, fake, ws, None) == 1
    # paged layout needs max_pages / num_pages
    dp = mod.Dims(max_ctx=1024, pool_blocks=64, topk=128, max_pages=0, num_pages=0)
    assert lib.indexer_full_topk(ctypes.byref(dp.c()), 1, fake, fake, *([fake] * 6), fake,
                                 mod.workspace_size(dp, 1), None) == 1
    # an indexer-K cache beyond 32-bit row coordinates (4096 x 2^20 rows; paged:
    # 2^26 pages of 64) is an unsupported shape, reported before the workspace is read
    dbig = mod.Dims(max_ctx=1 << 20)
    assert lib.indexer_full_topk(ctypes.byref(dbig.c()), 4096, *args, fake, 1 << 40, None) == 2
    assert lib.indexer_reindex_topk(ctypes.byref(dbig.c()), 4096, fake, None, *([fake] * 5), fake, fake,
                                    1 << 40, None) == 2
    dpb = mod.Dims(max_ctx=1 << 20, max_pages=1 << 14, num_pages=1 << 26)
    assert lib.indexer_full_topk(ctypes.byref(dpb.c()), 1, fake, fake, *([fake] * 6), fake, 1 << 40,
                                 None) == 2
    # 2047 x 2^20 rows fit: the call gets past the row check and stops at the
    # misaligned workspace (before anything is launched)
    assert lib.indexer_full_topk(ctypes.byref(dbig.c()), 2047, *args, P(0x10010), 1 << 40, None) == 1
    assert lib.csa2_get_device_status(None, None, None) == 1
    assert lib.csa2_clear_device_status(None, None) == 1
    # the timeout self-test validates its arguments before launching
    assert lib.csa2_selftest_wait_timeout(None, 256, 1000, None) == 1
    assert lib.csa2_selftest_wait_timeout(P(0x10010), 256, 1000, None) == 1     # misaligned
    assert lib.csa2_selftest_wait_timeout(fake, 255, 1000, None) == 1
    assert lib.csa2_selftest_wait_timeout(fake, 256, 0, None) == 1
    assert lib.csa2_selftest_wait_timeout(fake, 256, 2000000, None) == 1


def test_workspace_layout_mirror(mod):
    """The test-side mirror of the workspace layout agrees with the library's size."""
    from tests.helpers import ws_offsets
    d = mod.Dims(max_ctx=4096, pool_blocks=64, topk=128)
    off = ws_offsets(d, 3)
    assert off["blk_delta"] > off["blk_scores"] > off["pos_scores"] >= 256
    assert mod.workspace_size(d, 3) > off["ri_delta"]


def test_host_argument_errors_fp4_and_multi_query(mod):
    """The FP4 indexer-key write, the FP4 indexer dtype and the multi-query
    attention call validate on the host, before any CUDA call."""
    lib = mod._lib
    P = ctypes.c_void_p
    fake = P(0x10000)
    # FP4 indexer-key write: null / negative / misaligned / too many rows without destinations
    assert lib.fp4_idx_k_quantize_scatter(None, 4, None, fake, 16, None) == 1
    assert lib.fp4_idx_k_quantize_scatter(fake, -1, None, fake, 16, None) == 1
    assert lib.fp4_idx_k_quantize_scatter(fake, 4, None, fake, -1, None) == 1
    assert lib.fp4_idx_k_quantize_scatter(P(0x10008), 4, None, fake, 16, None) == 1
    assert lib.fp4_idx_k_quantize_scatter(fake, 4, None, P(0x10008), 16, None) == 1
    assert lib.fp4_idx_k_quantize_scatter(fake, 4, P(0x10004), fake, 16, None) == 1
    assert lib.fp4_idx_k_quantize_scatter(fake, 17, None, fake, 16, None) == 1
    assert lib.fp4_idx_k_quantize_scatter(None, 0, None, None, 0, None) == 0      # empty: no-op
    # FP4 indexer dims: idx_dim must be 128; the FP4 query must be 16-byte aligned
    d4 = mod.Dims(idx_k_dtype=mod.IDXK_FP4, max_ctx=1024, pool_blocks=64, topk=128)
    assert mod.workspace_size(d4, 2) > 0
    with pytest.raises(mod.Csa2Error) as e:
        mod.workspace_size(mod.Dims(idx_k_dtype=mod.IDXK_FP4, idx_dim=64), 1)
    assert e.value.code == 2
    ws = mod.workspace_size(d4, 2)
    wsp = P(0x20000)
    args = [fake, None, fake, P(0x10004)] + [fake] * 4      # idx_q only 4-byte aligned
    assert lib.indexer_full_topk(ctypes.byref(d4.c()), 2, *args, wsp, ws, None) == 1
    # multi-query attention: q_len outside 1..4, more than 8 chunks with q_len > 1, bad mode
    d = mod.Dims(max_ctx=1024, pool_blocks=64, topk=512)
    dc = ctypes.byref(d.c())
    wsa = mod.workspace_size(d, 2)
    a = [fake] * 4 + [None] + [fake] * 4
    for ql in (0, 5, -1):
        assert lib.csa2_sparse_attn_decode_mq(dc, 2, ql, 0, *a, 0.1, fake, fake, wsp, wsa, None) == 2
    dbig = mod.Dims(max_ctx=4096, pool_blocks=64, topk=1024)
    wsb = mod.workspace_size(dbig, 2)
    assert lib.csa2_sparse_attn_decode_mq(ctypes.byref(dbig.c()), 2, 2, 0, *a, 0.1, fake, fake, wsp, wsb,
                                          None) == 2
    assert lib.csa2_sparse_attn_decode_mq(dc, 2, 2, 3, *a, 0.1, fake, fake, wsp, wsa, None) == 1
    assert lib.csa2_sparse_attn_decode_mq(dc, 2, 2, 0, *a, float("nan"), fake, fake, wsp, wsa, None) == 1
    # q_len 1 with more than 8 chunks stays allowed (the split-KV path): it gets past the
    # shape checks and stops at the misaligned workspace
    assert lib.csa2_sparse_attn_decode_mq(ctypes.byref(dbig.c()), 2, 1, 0, *a, 0.1, fake, fake, P(0x20010),
                                          wsb, None) == 1


def test_indexer_ex_flags(mod):
    lib = mod._lib
    P = ctypes.c_void_p
    fake = P(0x10000)
    d = mod.Dims(max_ctx=1024, pool_blocks=64, topk=128)
    ws = mod.workspace_size(d, 2)
    args = [fake, None] + [fake] * 6
    assert lib.indexer_full_topk_ex(ctypes.byref(d.c()), 2, 2, *args, fake, ws, None) == 1      # unknown flag
    assert lib.indexer_full_topk_ex(ctypes.byref(d.c()), 2, 1, *args, fake, ws - 1, None) == 3   # checks as usual
    assert lib.indexer_reindex_topk_ex(ctypes.byref(d.c()), 2, -1, fake, None, *([fake] * 6), fake, ws, None) == 1


def test_kv_append_ex_flags(mod):
    lib = mod._lib
    P = ctypes.c_void_p
    fake = P(0x10000)
    f = lib.fp4_kv_quantize_scatter_ex
    assert f(fake, 4, fake, fake, fake, 2, None) == 1          # unknown flag
    assert f(fake, 4, fake, fake, fake, -1, None) == 1
    assert f(fake, 0, fake, fake, fake, 1, None) == 0          # nothing to write
    assert f(None, 4, fake, fake, fake, 1, None) == 1          # checks as usual
    assert f(P(0x10008), 4, fake, fake, fake, 1, None) == 1    # x not 16-byte aligned
    assert mod.KV_EARLY_INPUTS == 1
