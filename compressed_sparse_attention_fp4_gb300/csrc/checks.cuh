// checks.cuh -- host-side argument checks shared by the library's entry points
// (api.cu, noalloc.cu).  Every check returns a status without touching the
// device; an entry point returns it before launching anything.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace csa2 {

inline bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The fields of csa2_dims that the attention kernels read.
inline csa2_status check_attn_dims(const csa2_dims* d, int32_t batch) {
  if (!d || batch < 0) return CSA2_ERR_INVALID_ARG;
  if (d->topk < 1 || d->topk > kMaxTopk) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (d->heads < 1 || d->heads > kMaxHeads) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (d->swa < 0 || d->swa > kMaxSwa) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (d->max_ctx < 1 || d->max_ctx > kMaxCtx) return CSA2_ERR_UNSUPPORTED_SHAPE;
  return CSA2_OK;
}

// Every field of csa2_dims (the indexer calls and the workspace layout).
inline csa2_status check_dims(const csa2_dims* d, int32_t batch) {
  csa2_status st = check_attn_dims(d, batch);
  if (st != CSA2_OK) return st;
  if (d->idx_k_dtype != CSA2_IDXK_E4M3 && d->idx_k_dtype != CSA2_IDXK_F32 && d->idx_k_dtype != CSA2_IDXK_FP4)
    return CSA2_ERR_INVALID_ARG;
  if (d->idx_heads < 1 || d->idx_heads > kMaxIdxHeads) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (d->idx_k_dtype != CSA2_IDXK_F32 && d->idx_dim != 128) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (d->idx_k_dtype == CSA2_IDXK_F32 && d->idx_dim != 64) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (d->pool_blocks < 1 || d->pool_blocks > kMaxPool) return CSA2_ERR_UNSUPPORTED_SHAPE;
  return CSA2_OK;
}

// A paged cache: page-table geometry and alignment.
inline csa2_status check_paging(const csa2_dims* d, const int32_t* page_table) {
  if (!page_table) return CSA2_OK;
  if (d->max_pages < 1 || d->num_pages < 1) return CSA2_ERR_INVALID_ARG;
  if (int64_t(d->max_pages) * kPage > kMaxCtx) return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (!is_aligned(page_table, 4)) return CSA2_ERR_INVALID_ARG;
  return CSA2_OK;
}

// Pointers of an attention call (batch > 0): presence and alignment.
inline csa2_status check_attn_ptrs(const csa2_dims* d, int32_t mode, const uint16_t* q, const uint8_t* kv_codes,
                                   const uint8_t* kv_scales, const uint16_t* kv_rope, const int32_t* ctx_len,
                                   const int32_t* topk, const uint16_t* swa_kv, const int32_t* swa_len,
                                   float scale, const float* out, const float* lse) {
  if (mode < CSA2_MODE_FULL || mode > CSA2_MODE_REUSE) return CSA2_ERR_INVALID_ARG;
  if (!q || !kv_codes || !kv_scales || !kv_rope || !ctx_len || !topk || !swa_len || !out || !lse)
    return CSA2_ERR_INVALID_ARG;
  if (d->swa > 0 && !swa_kv) return CSA2_ERR_INVALID_ARG;
  if (!is_aligned(kv_codes, 16) || !is_aligned(kv_scales, 2) || !is_aligned(kv_rope, 16) || !is_aligned(q, 16) ||
      !is_aligned(out, 16) || (swa_kv && !is_aligned(swa_kv, 16)))
    return CSA2_ERR_INVALID_ARG;
  if (!(scale == scale)) return CSA2_ERR_INVALID_ARG;
  return CSA2_OK;
}

}  // namespace csa2
