"""Python binding of libcsa2.so, the GB300 CSA2 decode hot-path library.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory and streams; tensors are passed by
``data_ptr()`` and the current CUDA stream.  The names follow the C ABI in
``include/csa2.h``.  Importing this module loads the library and raises if it
is missing -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))  # package directory
LIB_PATH = os.path.join(_PKG, "_build", "libcsa2.so")

LATENT, ROPE, DQK, PAGE, BLOCK = 512, 64, 576, 64, 8
IDXK_E4M3, IDXK_F32, IDXK_FP4 = 0, 1, 2
MODE_FULL, MODE_REINDEX, MODE_REUSE = 0, 1, 2
MAX_QLEN = 4
IDX_EARLY_INPUTS = 1
KV_EARLY_INPUTS = 1

STATUS = {0: "CSA2_OK", 1: "CSA2_ERR_INVALID_ARG", 2: "CSA2_ERR_UNSUPPORTED_SHAPE",
          3: "CSA2_ERR_WORKSPACE_TOO_SMALL", 4: "CSA2_ERR_CUDA",
          5: "CSA2_ERR_DEVICE_ASSERT", 6: "CSA2_ERR_TIMEOUT"}

# exported symbols and their ctypes signatures
_P, _I32, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float


class CKernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int32), ("total_ms", ctypes.c_double)]


class CDims(ctypes.Structure):
    _fields_ = [("idx_heads", ctypes.c_int32), ("idx_dim", ctypes.c_int32),
                ("idx_k_dtype", ctypes.c_int32), ("pool_blocks", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("heads", ctypes.c_int32), ("swa", ctypes.c_int32),
                ("max_pages", ctypes.c_int32), ("num_pages", ctypes.c_int64),
                ("max_ctx", ctypes.c_int64)]


SIGNATURES = {
    "csa2_version": (_I32, []),
    "csa2_status_string": (ctypes.c_char_p, [_I32]),
    "csa2_workspace_size": (_I32, [ctypes.POINTER(CDims), _I32, ctypes.POINTER(_SZ)]),
    "fp4_kv_quantize": (_I32, [_P, _I64, _P, _P, _P]),
    "fp4_kv_quantize_scatter": (_I32, [_P, _I64, _P, _P, _P, _P]),
    "fp4_kv_quantize_scatter_ex": (_I32, [_P, _I64, _P, _P, _P, _I32, _P]),
    "fp4_idx_k_quantize_scatter": (_I32, [_P, _I64, _P, _P, _I64, _P]),
    "fp4_kv_dequantize": (_I32, [_P, _P, _I64, _P, _P]),
    "indexer_full_topk": (_I32, [ctypes.POINTER(CDims), _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                                 _P, _SZ, _P]),
    "indexer_reindex_topk": (_I32, [ctypes.POINTER(CDims), _I32, _P, _P, _P, _P, _P, _P, _P,
                                    _P, _P, _SZ, _P]),
    "indexer_full_topk_ex": (_I32, [ctypes.POINTER(CDims), _I32, _I32, _P, _P, _P, _P, _P, _P, _P,
                                    _P, _P, _SZ, _P]),
    "indexer_reindex_topk_ex": (_I32, [ctypes.POINTER(CDims), _I32, _I32, _P, _P, _P, _P, _P, _P,
                                       _P, _P, _P, _SZ, _P]),
    "csa2_sparse_attn_decode": (_I32, [ctypes.POINTER(CDims), _I32, _I32, _P, _P, _P, _P, _P,
                                       _P, _P, _P, _P, _F, _P, _P, _P, _SZ, _P]),
    "csa2_sparse_attn_decode_mq": (_I32, [ctypes.POINTER(CDims), _I32, _I32, _I32, _P, _P, _P, _P, _P,
                                          _P, _P, _P, _P, _F, _P, _P, _P, _SZ, _P]),
    "csa2_sparse_attn_decode_noalloc": (_I32, [ctypes.POINTER(CDims), _I32, _I32, _P, _P, _P, _P,
                                               _P, _P, _P, _P, _P, _F, _P, _P, _P, _P]),
    "csa2_get_device_status": (_I32, [_P, _P, ctypes.POINTER(_I32)]),
    "csa2_profile_enable": (_I32, [_I32]),
    "csa2_profile_read": (_I32, [ctypes.POINTER(CKernelTime), _I32, ctypes.POINTER(_I32)]),
    "csa2_clear_device_status": (_I32, [_P, _P]),
    "csa2_selftest_wait_timeout": (_I32, [_P, _SZ, ctypes.c_uint32, _P]),
}


class Csa2Error(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libcsa2.so not built ({path}); run __graft_entry__.build() or "
                          "python -m compressed_sparse_attention_fp4_gb300.build")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = load_library()


def _check(name: str, code: int):
    if code != 0:
        raise Csa2Error(name, code)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


@dataclass
class Dims:
    """Python view of ``csa2_dims`` (see include/csa2.h)."""
    idx_heads: int = 16
    idx_dim: int = 128
    idx_k_dtype: int = IDXK_E4M3
    pool_blocks: int = 2048
    topk: int = 512
    heads: int = 64
    swa: int = 128
    max_pages: int = 0
    num_pages: int = 0
    max_ctx: int = 131072

    def c(self) -> CDims:
        return CDims(self.idx_heads, self.idx_dim, self.idx_k_dtype, self.pool_blocks,
                     self.topk, self.heads, self.swa, self.max_pages, self.num_pages,
                     self.max_ctx)


def version() -> int:
    return _lib.csa2_version()


def workspace_size(dims: Dims, batch: int) -> int:
    out = ctypes.c_size_t(0)
    _check("csa2_workspace_size", _lib.csa2_workspace_size(ctypes.byref(dims.c()), batch, ctypes.byref(out)))
    return out.value


def alloc_workspace(dims: Dims, batch: int, device="cuda") -> torch.Tensor:
    """Zeroed workspace tensor (uint8, 256-byte aligned by the allocator)."""
    return torch.zeros(workspace_size(dims, batch), dtype=torch.uint8, device=device)


def fp4_kv_quantize(x: torch.Tensor, codes: torch.Tensor | None = None,
                    scales: torch.Tensor | None = None, stream=None):
    """bf16 [n, 512] -> (codes uint8 [n, 256], scales uint8 [n, 32])."""
    n = x.shape[0]
    if codes is None:
        codes = torch.empty((n, LATENT // 2), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((n, LATENT // 16), dtype=torch.uint8, device=x.device)
    _check("fp4_kv_quantize", _lib.fp4_kv_quantize(_ptr(x), n, _ptr(codes), _ptr(scales), _stream(stream)))
    return codes, scales


def fp4_kv_quantize_scatter(x: torch.Tensor, dst_rows: torch.Tensor, codes: torch.Tensor,
                            scales: torch.Tensor, stream=None, flags: int = 0):
    """Quantize row i of x into cache row dst_rows[i] (int64).  flags:
    KV_EARLY_INPUTS (see fp4_kv_quantize_scatter_ex in include/csa2.h) or 0."""
    if flags:
        _check("fp4_kv_quantize_scatter_ex",
               _lib.fp4_kv_quantize_scatter_ex(_ptr(x), x.shape[0], _ptr(dst_rows), _ptr(codes),
                                               _ptr(scales), int(flags), _stream(stream)))
        return
    _check("fp4_kv_quantize_scatter",
           _lib.fp4_kv_quantize_scatter(_ptr(x), x.shape[0], _ptr(dst_rows), _ptr(codes),
                                        _ptr(scales), _stream(stream)))


def fp4_idx_k_quantize_scatter(x: torch.Tensor, idx_k: torch.Tensor, cache_rows: int,
                               dst_rows: torch.Tensor | None = None, stream=None):
    """bf16 [n, 128] indexer keys into the two-plane FP4 indexer-K buffer
    ``idx_k`` (uint8, cache_rows * 72 bytes: codes [rows][64], then scales
    [rows][8]); row i goes to dst_rows[i] (int64) or to row i."""
    _check("fp4_idx_k_quantize_scatter",
           _lib.fp4_idx_k_quantize_scatter(_ptr(x), x.shape[0], _ptr(dst_rows), _ptr(idx_k), int(cache_rows),
                                           _stream(stream)))


def fp4_idx_k_planes(idx_k: torch.Tensor, cache_rows: int):
    """Views (codes [rows, 64], scales [rows, 8]) of a two-plane FP4 indexer-K buffer."""
    flat = idx_k.reshape(-1)
    return (flat[:cache_rows * 64].view(cache_rows, 64),
            flat[cache_rows * 64:cache_rows * 72].view(cache_rows, 8))


def fp4_kv_dequantize(codes: torch.Tensor, scales: torch.Tensor, y: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """(codes, scales) -> bf16 [n, 512]."""
    n = codes.shape[0]
    if y is None:
        y = torch.empty((n, LATENT), dtype=torch.bfloat16, device=codes.device)
    _check("fp4_kv_dequantize", _lib.fp4_kv_dequantize(_ptr(codes), _ptr(scales), n, _ptr(y), _stream(stream)))
    return y


def indexer_full_topk(dims: Dims, batch: int, idx_k, page_table, ctx_len, idx_q, w,
                      pool_out, pool_len_out, topk_out, ws, stream=None, flags: int = 0):
    """flags: IDX_EARLY_INPUTS (see indexer_full_topk_ex in include/csa2.h) or 0."""
    if flags:
        _check("indexer_full_topk_ex", _lib.indexer_full_topk_ex(
            ctypes.byref(dims.c()), batch, int(flags), _ptr(idx_k), _ptr(page_table), _ptr(ctx_len),
            _ptr(idx_q), _ptr(w), _ptr(pool_out), _ptr(pool_len_out), _ptr(topk_out), _ptr(ws), ws.numel(),
            _stream(stream)))
        return
    _check("indexer_full_topk", _lib.indexer_full_topk(
        ctypes.byref(dims.c()), batch, _ptr(idx_k), _ptr(page_table), _ptr(ctx_len), _ptr(idx_q),
        _ptr(w), _ptr(pool_out), _ptr(pool_len_out), _ptr(topk_out), _ptr(ws), ws.numel(),
        _stream(stream)))


def indexer_reindex_topk(dims: Dims, batch: int, idx_k, page_table, ctx_len, idx_q, w,
                         pool_blocks, pool_len, topk_out, ws, stream=None, flags: int = 0):
    """flags: IDX_EARLY_INPUTS (see indexer_reindex_topk_ex in include/csa2.h) or 0."""
    if flags:
        _check("indexer_reindex_topk_ex", _lib.indexer_reindex_topk_ex(
            ctypes.byref(dims.c()), batch, int(flags), _ptr(idx_k), _ptr(page_table), _ptr(ctx_len),
            _ptr(idx_q), _ptr(w), _ptr(pool_blocks), _ptr(pool_len), _ptr(topk_out), _ptr(ws), ws.numel(),
            _stream(stream)))
        return
    _check("indexer_reindex_topk", _lib.indexer_reindex_topk(
        ctypes.byref(dims.c()), batch, _ptr(idx_k), _ptr(page_table), _ptr(ctx_len), _ptr(idx_q),
        _ptr(w), _ptr(pool_blocks), _ptr(pool_len), _ptr(topk_out), _ptr(ws), ws.numel(),
        _stream(stream)))


def csa2_sparse_attn_decode(dims: Dims, batch: int, mode: int, q, kv_codes, kv_scales, kv_rope,
                            page_table, ctx_len, topk, swa_kv, swa_len, scale: float, out, lse,
                            ws, stream=None):
    _check("csa2_sparse_attn_decode", _lib.csa2_sparse_attn_decode(
        ctypes.byref(dims.c()), batch, mode, _ptr(q), _ptr(kv_codes), _ptr(kv_scales),
        _ptr(kv_rope), _ptr(page_table), _ptr(ctx_len), _ptr(topk), _ptr(swa_kv), _ptr(swa_len),
        float(scale), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))


def csa2_sparse_attn_decode_mq(dims: Dims, batch: int, q_len: int, mode: int, q, kv_codes, kv_scales,
                               kv_rope, page_table, ctx_len, topk, swa_kv, swa_len, scale: float, out, lse,
                               ws, stream=None):
    """Multi-query decode attention: q bf16 [B, q_len, H, 576] (the newest
    q_len tokens, oldest first), out fp32 [B, q_len, H, 512], lse [B, q_len, H]."""
    _check("csa2_sparse_attn_decode_mq", _lib.csa2_sparse_attn_decode_mq(
        ctypes.byref(dims.c()), batch, int(q_len), mode, _ptr(q), _ptr(kv_codes), _ptr(kv_scales),
        _ptr(kv_rope), _ptr(page_table), _ptr(ctx_len), _ptr(topk), _ptr(swa_kv), _ptr(swa_len),
        float(scale), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))


def csa2_sparse_attn_decode_noalloc(dims: Dims, batch: int, mode: int, q, kv_codes, kv_scales,
                                    kv_rope, page_table, ctx_len, topk, swa_kv, swa_len,
                                    scale: float, out, lse, err_word=None, stream=None):
    """Decode attention without a workspace: for callers that cannot allocate.

    The split-KV scratch is a fixed array inside the library (12 MiB per GPU,
    kept until exit); calls that overlap on the GPU race on it.  err_word is
    an optional device int32 tensor that receives the call's device error bits.
    """
    _check("csa2_sparse_attn_decode_noalloc", _lib.csa2_sparse_attn_decode_noalloc(
        ctypes.byref(dims.c()), batch, mode, _ptr(q), _ptr(kv_codes), _ptr(kv_scales),
        _ptr(kv_rope), _ptr(page_table), _ptr(ctx_len), _ptr(topk), _ptr(swa_kv), _ptr(swa_len),
        float(scale), _ptr(out), _ptr(lse), _ptr(err_word), _stream(stream)))


def get_device_status(ws: torch.Tensor, stream=None) -> int:
    """The workspace's device error word (synchronises the stream)."""
    word = ctypes.c_int32(0)
    code = _lib.csa2_get_device_status(_ptr(ws), _stream(stream), ctypes.byref(word))
    if code not in (0, 5, 6):
        raise Csa2Error("csa2_get_device_status", code)
    return word.value


def profile_enable(on: bool = True):
    """Bracket every library kernel launch with CUDA events (not during capture)."""
    _check("csa2_profile_enable", _lib.csa2_profile_enable(1 if on else 0))


def profile_read() -> dict:
    """{kernel name: (launches, total ms)} of the launches recorded so far."""
    arr = (CKernelTime * 64)()
    n = ctypes.c_int32(0)
    _check("csa2_profile_read", _lib.csa2_profile_read(arr, 64, ctypes.byref(n)))
    return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(min(n.value, 64))}


def clear_device_status(ws: torch.Tensor, stream=None):
    _check("csa2_clear_device_status", _lib.csa2_clear_device_status(_ptr(ws), _stream(stream)))


def selftest_wait_timeout(ws: torch.Tensor, limit_us: int = 2000, stream=None):
    """Runs the device timeout path on purpose: a bounded wait on an mbarrier
    nothing arrives at gives up after limit_us and sets CSA2_DEV_TIMEOUT in
    the error word of ws (read it with get_device_status)."""
    _check("csa2_selftest_wait_timeout",
           _lib.csa2_selftest_wait_timeout(_ptr(ws), ws.numel(), int(limit_us), _stream(stream)))
