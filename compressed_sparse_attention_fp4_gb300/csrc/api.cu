// api.cu -- the extern "C" boundary of libcsa2.so: argument checks, workspace
// layout and kernel launches.  Every call validates on the host and returns a
// status without launching anything when an argument is wrong.
#include <cstdint>

#include "checks.cuh"
#include "kernels.cuh"

using namespace csa2;

namespace {

inline bool aligned(const void* p, uintptr_t a) { return is_aligned(p, a); }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

csa2_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA; }

// Rows of the indexer-K cache: B * max_ctx contiguous, num_pages * 64 paged.
int64_t idx_cache_rows(const csa2_dims* d, int32_t batch, const int32_t* page_table) {
  return page_table ? d->num_pages * int64_t(kPage) : int64_t(batch) * d->max_ctx;
}

// The indexer scan addresses cache rows with 32-bit tensor coordinates.
csa2_status check_idx_rows(const csa2_dims* d, int32_t batch, const int32_t* page_table) {
  return idx_cache_rows(d, batch, page_table) > int64_t(INT32_MAX) ? CSA2_ERR_UNSUPPORTED_SHAPE : CSA2_OK;
}

// Pointer checks of an indexer call; the FP4 query is read in 16-byte pieces.
csa2_status check_idx_ptrs(const csa2_dims* d, const void* idx_k, const void* idx_q) {
  if (!aligned(idx_k, 16) || !aligned(idx_q, d->idx_k_dtype == CSA2_IDXK_FP4 ? 16 : 4)) return CSA2_ERR_INVALID_ARG;
  return CSA2_OK;
}

const uint8_t* fp4_scales_plane(const csa2_dims* d, int32_t batch, const int32_t* page_table, const void* idx_k) {
  if (d->idx_k_dtype != CSA2_IDXK_FP4) return nullptr;
  return static_cast<const uint8_t*>(idx_k) + idx_cache_rows(d, batch, page_table) * 64;
}

csa2_status check_ws(const csa2_dims* d, int32_t batch, const void* ws, size_t ws_bytes, WsLayout* L) {
  *L = make_layout(*d, batch);
  if (!ws || !aligned(ws, 256)) return CSA2_ERR_INVALID_ARG;
  if (ws_bytes < size_t(L->total)) return CSA2_ERR_WORKSPACE_TOO_SMALL;
  return CSA2_OK;
}

// Attention call with q_len queries per sequence (1: the single-query call).
csa2_status attn_call(const csa2_dims* d, int32_t batch, int32_t q_len, int32_t mode, const uint16_t* q,
                      const uint8_t* kv_codes, const uint8_t* kv_scales, const uint16_t* kv_rope,
                      const int32_t* page_table, const int32_t* ctx_len, const int32_t* topk,
                      const uint16_t* swa_kv, const int32_t* swa_len, float scale, float* out, float* lse, void* ws,
                      size_t ws_bytes, void* stream) {
  csa2_status st = check_dims(d, batch);
  if (st != CSA2_OK) return st;
  if (mode < CSA2_MODE_FULL || mode > CSA2_MODE_REUSE) return CSA2_ERR_INVALID_ARG;
  if (q_len < 1 || q_len > CSA2_MAX_QLEN) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (q_len > 1 && attn_uses_partials(*d)) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if ((st = check_paging(d, page_table)) != CSA2_OK) return st;
  WsLayout L;
  if ((st = check_ws(d, batch, ws, ws_bytes, &L)) != CSA2_OK) return st;
  if (batch == 0) return CSA2_OK;
  if ((st = check_attn_ptrs(d, mode, q, kv_codes, kv_scales, kv_rope, ctx_len, topk, swa_kv, swa_len, scale, out,
                            lse)) != CSA2_OK)
    return st;
  AttnArgs a = {};
  a.d = *d;
  a.batch = batch;
  a.q = q;
  a.codes = kv_codes;
  a.scales = kv_scales;
  a.rope = kv_rope;
  a.page_table = page_table;
  a.ctx_len = ctx_len;
  a.topk = topk;
  a.swa = swa_kv;
  a.swa_len = swa_len;
  a.scale = scale;
  a.out = out;
  a.lse = lse;
  a.ws = static_cast<uint8_t*>(ws);
  a.L = L;
  a.early = mode == CSA2_MODE_REUSE;
  a.q_len = q_len;
  return from_cuda(launch_attention(a, as_stream(stream)));
}

}  // namespace

extern "C" {

int32_t csa2_version(void) { return 100; }

const char* csa2_status_string(csa2_status st) {
  switch (st) {
    case CSA2_OK: return "CSA2_OK";
    case CSA2_ERR_INVALID_ARG: return "CSA2_ERR_INVALID_ARG";
    case CSA2_ERR_UNSUPPORTED_SHAPE: return "CSA2_ERR_UNSUPPORTED_SHAPE";
    case CSA2_ERR_WORKSPACE_TOO_SMALL: return "CSA2_ERR_WORKSPACE_TOO_SMALL";
    case CSA2_ERR_CUDA: return "CSA2_ERR_CUDA";
    case CSA2_ERR_DEVICE_ASSERT: return "CSA2_ERR_DEVICE_ASSERT";
    case CSA2_ERR_TIMEOUT: return "CSA2_ERR_TIMEOUT";
  }
  return "CSA2_ERR_UNKNOWN";
}

csa2_status csa2_workspace_size(const csa2_dims* d, int32_t batch, size_t* bytes) {
  if (!bytes) return CSA2_ERR_INVALID_ARG;
  csa2_status st = check_dims(d, batch);
  if (st != CSA2_OK) return st;
  *bytes = size_t(make_layout(*d, batch).total);
  return CSA2_OK;
}

csa2_status fp4_kv_quantize(const uint16_t* x, int64_t n, uint8_t* codes, uint8_t* scales,
                            void* stream) {
  if (n < 0) return CSA2_ERR_INVALID_ARG;
  if (n == 0) return CSA2_OK;
  if (!x || !codes || !scales || !aligned(x, 16) || !aligned(codes, 4)) return CSA2_ERR_INVALID_ARG;
  return from_cuda(launch_quantize(x, n, nullptr, codes, scales, false, as_stream(stream)));
}

csa2_status fp4_kv_quantize_scatter_ex(const uint16_t* x, int64_t n, const int64_t* dst_rows,
                                       uint8_t* codes, uint8_t* scales, int32_t flags, void* stream) {
  if (n < 0 || (flags & ~int32_t(CSA2_KV_EARLY_INPUTS)) != 0) return CSA2_ERR_INVALID_ARG;
  if (n == 0) return CSA2_OK;
  if (!x || !dst_rows || !codes || !scales || !aligned(x, 16) || !aligned(codes, 4) ||
      !aligned(dst_rows, 8))
    return CSA2_ERR_INVALID_ARG;
  return from_cuda(launch_quantize(x, n, dst_rows, codes, scales, (flags & CSA2_KV_EARLY_INPUTS) != 0,
                                   as_stream(stream)));
}

csa2_status fp4_kv_quantize_scatter(const uint16_t* x, int64_t n, const int64_t* dst_rows,
                                    uint8_t* codes, uint8_t* scales, void* stream) {
  return fp4_kv_quantize_scatter_ex(x, n, dst_rows, codes, scales, 0, stream);
}

csa2_status fp4_idx_k_quantize_scatter(const uint16_t* x, int64_t n, const int64_t* dst_rows,
                                       uint8_t* idx_k, int64_t cache_rows, void* stream) {
  if (n < 0 || cache_rows < 0) return CSA2_ERR_INVALID_ARG;
  if (n == 0) return CSA2_OK;
  if (!x || !idx_k || !aligned(x, 16) || !aligned(idx_k, 16) || (dst_rows && !aligned(dst_rows, 8)))
    return CSA2_ERR_INVALID_ARG;
  if (!dst_rows && n > cache_rows) return CSA2_ERR_INVALID_ARG;
  return from_cuda(launch_quantize_idx(x, n, dst_rows, idx_k, cache_rows, as_stream(stream)));
}

csa2_status fp4_kv_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t n, uint16_t* y,
                              void* stream) {
  if (n < 0) return CSA2_ERR_INVALID_ARG;
  if (n == 0) return CSA2_OK;
  if (!codes || !scales || !y || !aligned(codes, 8) || !aligned(y, 16)) return CSA2_ERR_INVALID_ARG;
  return from_cuda(launch_dequantize(codes, scales, n, y, as_stream(stream)));
}

csa2_status indexer_full_topk(const csa2_dims* d, int32_t batch, const void* idx_k,
                              const int32_t* page_table, const int32_t* ctx_len, const void* idx_q,
                              const float* w, int32_t* pool_blocks_out, int32_t* pool_len_out,
                              int32_t* topk_out, void* ws, size_t ws_bytes, void* stream) {
  return indexer_full_topk_ex(d, batch, 0, idx_k, page_table, ctx_len, idx_q, w, pool_blocks_out, pool_len_out,
                              topk_out, ws, ws_bytes, stream);
}

csa2_status indexer_full_topk_ex(const csa2_dims* d, int32_t batch, int32_t flags, const void* idx_k,
                                 const int32_t* page_table, const int32_t* ctx_len, const void* idx_q,
                                 const float* w, int32_t* pool_blocks_out, int32_t* pool_len_out,
                                 int32_t* topk_out, void* ws, size_t ws_bytes, void* stream) {
  if (flags & ~int32_t(CSA2_IDX_EARLY_INPUTS)) return CSA2_ERR_INVALID_ARG;
  csa2_status st = check_dims(d, batch);
  if (st != CSA2_OK) return st;
  if ((st = check_paging(d, page_table)) != CSA2_OK) return st;
  if ((st = check_idx_rows(d, batch, page_table)) != CSA2_OK) return st;
  WsLayout L;
  if ((st = check_ws(d, batch, ws, ws_bytes, &L)) != CSA2_OK) return st;
  if (batch == 0) return CSA2_OK;
  if (!idx_k || !ctx_len || !idx_q || !w || !pool_blocks_out || !pool_len_out || !topk_out)
    return CSA2_ERR_INVALID_ARG;
  if ((st = check_idx_ptrs(d, idx_k, idx_q)) != CSA2_OK) return st;
  IdxArgs a = {};
  a.d = *d;
  a.batch = batch;
  a.idx_k = idx_k;
  a.idx_scales = fp4_scales_plane(d, batch, page_table, idx_k);
  a.page_table = page_table;
  a.ctx_len = ctx_len;
  a.idx_q = idx_q;
  a.w = w;
  a.pool_out = pool_blocks_out;
  a.pool_len_out = pool_len_out;
  a.topk_out = topk_out;
  a.ws = static_cast<uint8_t*>(ws);
  a.L = L;
  a.early = (flags & CSA2_IDX_EARLY_INPUTS) ? 1 : 0;
  return from_cuda(launch_full(a, as_stream(stream)));
}

csa2_status indexer_reindex_topk(const csa2_dims* d, int32_t batch, const void* idx_k,
                                 const int32_t* page_table, const int32_t* ctx_len,
                                 const void* idx_q, const float* w, const int32_t* pool_blocks,
                                 const int32_t* pool_len, int32_t* topk_out, void* ws,
                                 size_t ws_bytes, void* stream) {
  return indexer_reindex_topk_ex(d, batch, 0, idx_k, page_table, ctx_len, idx_q, w, pool_blocks, pool_len, topk_out,
                                 ws, ws_bytes, stream);
}

csa2_status indexer_reindex_topk_ex(const csa2_dims* d, int32_t batch, int32_t flags, const void* idx_k,
                                    const int32_t* page_table, const int32_t* ctx_len, const void* idx_q,
                                    const float* w, const int32_t* pool_blocks, const int32_t* pool_len,
                                    int32_t* topk_out, void* ws, size_t ws_bytes, void* stream) {
  if (flags & ~int32_t(CSA2_IDX_EARLY_INPUTS)) return CSA2_ERR_INVALID_ARG;
  csa2_status st = check_dims(d, batch);
  if (st != CSA2_OK) return st;
  if ((st = check_paging(d, page_table)) != CSA2_OK) return st;
  if ((st = check_idx_rows(d, batch, page_table)) != CSA2_OK) return st;
  WsLayout L;
  if ((st = check_ws(d, batch, ws, ws_bytes, &L)) != CSA2_OK) return st;
  if (batch == 0) return CSA2_OK;
  if (!idx_k || !ctx_len || !idx_q || !w || !pool_blocks || !pool_len || !topk_out)
    return CSA2_ERR_INVALID_ARG;
  if ((st = check_idx_ptrs(d, idx_k, idx_q)) != CSA2_OK) return st;
  IdxArgs a = {};
  a.d = *d;
  a.batch = batch;
  a.idx_k = idx_k;
  a.idx_scales = fp4_scales_plane(d, batch, page_table, idx_k);
  a.page_table = page_table;
  a.ctx_len = ctx_len;
  a.idx_q = idx_q;
  a.w = w;
  a.pool_in = pool_blocks;
  a.pool_len_in = pool_len;
  a.topk_out = topk_out;
  a.ws = static_cast<uint8_t*>(ws);
  a.L = L;
  a.early = (flags & CSA2_IDX_EARLY_INPUTS) ? 1 : 0;
  return from_cuda(launch_reindex(a, as_stream(stream)));
}

csa2_status csa2_sparse_attn_decode(const csa2_dims* d, int32_t batch, int32_t mode,
                                    const uint16_t* q, const uint8_t* kv_codes,
                                    const uint8_t* kv_scales, const uint16_t* kv_rope,
                                    const int32_t* page_table, const int32_t* ctx_len,
                                    const int32_t* topk, const uint16_t* swa_kv,
                                    const int32_t* swa_len, float scale, float* out, float* lse,
                                    void* ws, size_t ws_bytes, void* stream) {
  return attn_call(d, batch, 1, mode, q, kv_codes, kv_scales, kv_rope, page_table, ctx_len, topk, swa_kv, swa_len,
                   scale, out, lse, ws, ws_bytes, stream);
}

csa2_status csa2_sparse_attn_decode_mq(const csa2_dims* d, int32_t batch, int32_t q_len, int32_t mode,
                                       const uint16_t* q, const uint8_t* kv_codes,
                                       const uint8_t* kv_scales, const uint16_t* kv_rope,
                                       const int32_t* page_table, const int32_t* ctx_len,
                                       const int32_t* topk, const uint16_t* swa_kv,
                                       const int32_t* swa_len, float scale, float* out, float* lse,
                                       void* ws, size_t ws_bytes, void* stream) {
  return attn_call(d, batch, q_len, mode, q, kv_codes, kv_scales, kv_rope, page_table, ctx_len, topk, swa_kv,
                   swa_len, scale, out, lse, ws, ws_bytes, stream);
}

csa2_status csa2_get_device_status(const void* ws, void* stream, int32_t* word) {
  if (!ws || !word) return CSA2_ERR_INVALID_ARG;
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, as_stream(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return CSA2_ERR_CUDA;
  *word = v;
  if (v & CSA2_DEV_TIMEOUT) return CSA2_ERR_TIMEOUT;
  return v ? CSA2_ERR_DEVICE_ASSERT : CSA2_OK;
}

csa2_status csa2_clear_device_status(void* ws, void* stream) {
  if (!ws) return CSA2_ERR_INVALID_ARG;
  return from_cuda(cudaMemsetAsync(ws, 0, 256, as_stream(stream)));
}

}  // extern "C"
