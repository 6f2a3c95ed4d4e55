// noalloc.cu -- csa2_sparse_attn_decode_noalloc: the decode attention call
// for callers that cannot allocate GPU memory at all, not even a workspace.
//
// Some callers run inside another runtime's execution step (an engine plugin
// invoked at enqueue time, a real-time serving loop with a memory budget fixed
// up front) where calling cudaMalloc -- or asking their host for a buffer --
// is not allowed on the hot path.  For them this entry point keeps the
// split-KV scratch of the attention kernels in a fixed array that is part of
// the library image itself: a file-scope __device__ array, created when the
// library's module is loaded on a device and kept there until the process
// exits.  The caller still passes every input and output buffer.
//
// The array is shared by every call on a device and keeps the previous call's
// contents; the error word at its start is cleared by each call, the rest is
// fully rewritten before it is read.  Two calls whose work overlaps on the GPU
// (different streams, no ordering between them) race on the array.
#include <mutex>

#include "kernels.cuh"

using namespace csa2;

// The scratch.  Host code must not take this name as a device address: it
// only refers to the host-side shadow of the symbol.  The device address
// comes from cudaGetSymbolAddress below, once per device.
static __device__ __align__(256) uint8_t g_scratch[CSA2_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t kScratchBytes = CSA2_NOALLOC_SCRATCH_BYTES;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (set up on first use).
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

// OR the call's device error bits (first word of the scratch) into *err_word.
__global__ void publish_error_word(int32_t* err_word) {
  int32_t v = *reinterpret_cast<const int32_t*>(g_scratch);
  if (v) atomicOr(err_word, v);
}

inline bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" csa2_status csa2_sparse_attn_decode_noalloc(
    const csa2_dims* d, int32_t batch, int32_t mode, const uint16_t* q, const uint8_t* kv_codes,
    const uint8_t* kv_scales, const uint16_t* kv_rope, const int32_t* page_table,
    const int32_t* ctx_len, const int32_t* topk, const uint16_t* swa_kv, const int32_t* swa_len,
    float scale, float* out, float* lse, int32_t* err_word, void* stream) {
  if (!d || batch < 0) return CSA2_ERR_INVALID_ARG;
  if (mode < CSA2_MODE_FULL || mode > CSA2_MODE_REUSE) return CSA2_ERR_INVALID_ARG;
  if (d->heads < 1 || d->heads > kMaxHeads || d->topk < 1 || d->topk > kMaxTopk || d->swa < 0 ||
      d->swa > kMaxSwa || d->max_ctx < 1 || d->max_ctx > kMaxCtx)
    return CSA2_ERR_UNSUPPORTED_SHAPE;
  if (page_table && (d->max_pages < 1 || d->num_pages < 1 || !is_aligned(page_table, 4)))
    return CSA2_ERR_INVALID_ARG;
  // scratch needed: error word, partial outputs and (max, sum) per split
  WsLayout L = {};
  L.splits = (d->topk + d->swa + kAttnChunk - 1) / kAttnChunk;
  int64_t rows = int64_t(batch) * L.splits * d->heads;
  L.err = 0;
  L.attn_o = 256;
  L.attn_ml = align256(L.attn_o + rows * kLatent * 4);
  L.total = align256(L.attn_ml + rows * 2 * 4);
  if (L.total > int64_t(kScratchBytes)) return CSA2_ERR_WORKSPACE_TOO_SMALL;
  if (batch == 0) return CSA2_OK;
  if (!q || !kv_codes || !kv_scales || !kv_rope || !ctx_len || !topk || !swa_len || !out || !lse)
    return CSA2_ERR_INVALID_ARG;
  if (d->swa > 0 && !swa_kv) return CSA2_ERR_INVALID_ARG;
  if (!is_aligned(kv_codes, 16) || !is_aligned(kv_scales, 2) || !is_aligned(kv_rope, 16) || !is_aligned(q, 16) ||
      !is_aligned(out, 16) || (swa_kv && !is_aligned(swa_kv, 16)) ||
      (err_word && !is_aligned(err_word, 4)))
    return CSA2_ERR_INVALID_ARG;
  if (!(scale == scale)) return CSA2_ERR_INVALID_ARG;

  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return CSA2_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, 256, st) != cudaSuccess) return CSA2_ERR_CUDA;

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
  a.ws = static_cast<uint8_t*>(scratch);
  a.L = L;
  if (launch_attention(a, st) != cudaSuccess) return CSA2_ERR_CUDA;
  if (err_word) {
    publish_error_word<<<1, 1, 0, st>>>(err_word);
    if (cudaGetLastError() != cudaSuccess) return CSA2_ERR_CUDA;
  }
  return CSA2_OK;
}
