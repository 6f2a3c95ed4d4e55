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
// contents; the error word at its start is cleared by each call, the partial
// outputs (used only when Top-K + SWA exceeds 1024 entries) are fully
// rewritten before they are read.  Two calls whose work overlaps on the GPU
// (different streams, no ordering between them) race on the array.
#include <mutex>

#include "checks.cuh"
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

}  // namespace

extern "C" csa2_status csa2_sparse_attn_decode_noalloc(
    const csa2_dims* d, int32_t batch, int32_t mode, const uint16_t* q, const uint8_t* kv_codes,
    const uint8_t* kv_scales, const uint16_t* kv_rope, const int32_t* page_table,
    const int32_t* ctx_len, const int32_t* topk, const uint16_t* swa_kv, const int32_t* swa_len,
    float scale, float* out, float* lse, int32_t* err_word, void* stream) {
  csa2_status st = check_attn_dims(d, batch);
  if (st != CSA2_OK) return st;
  if (mode < CSA2_MODE_FULL || mode > CSA2_MODE_REUSE) return CSA2_ERR_INVALID_ARG;
  if ((st = check_paging(d, page_table)) != CSA2_OK) return st;
  // scratch needed: the error word; the partial outputs and (max, sum) per
  // chunk only when the chunks are merged by the combine kernel
  WsLayout L = {};
  L.splits = attn_splits(*d);
  L.err = 0;
  L.attn_o = 256;
  L.attn_ml = 256;
  L.total = 256;
  if (attn_uses_partials(*d)) {
    const int64_t rows = int64_t(batch) * L.splits * d->heads;
    L.attn_ml = align256(L.attn_o + rows * kLatent * 4);
    L.total = align256(L.attn_ml + rows * 2 * 4);
  }
  if (L.total > int64_t(kScratchBytes)) return CSA2_ERR_WORKSPACE_TOO_SMALL;
  if (batch == 0) return CSA2_OK;
  if ((st = check_attn_ptrs(d, mode, q, kv_codes, kv_scales, kv_rope, ctx_len, topk, swa_kv, swa_len, scale, out,
                            lse)) != CSA2_OK)
    return st;
  if (err_word && !is_aligned(err_word, 4)) return CSA2_ERR_INVALID_ARG;

  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return CSA2_ERR_CUDA;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, 256, cs) != cudaSuccess) return CSA2_ERR_CUDA;

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
  a.early = mode == CSA2_MODE_REUSE;
  a.q_len = 1;
  if (launch_attention(a, cs) != cudaSuccess) return CSA2_ERR_CUDA;
  if (err_word) {
    publish_error_word<<<1, 1, 0, cs>>>(err_word);
    if (cudaGetLastError() != cudaSuccess) return CSA2_ERR_CUDA;
  }
  return CSA2_OK;
}
