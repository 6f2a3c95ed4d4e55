// kernels.cuh -- argument blocks and host launchers of the library's kernels.
#pragma once

#include <atomic>

#include "common.cuh"

namespace csa2 {

// The function attributes a launcher has set, per device, so that each is
// set once per device and not on every call (the launch path of a decode
// step runs thousands of times a second).
constexpr int kMaxDevices = 64;
struct KernelAttrs {
  std::atomic<int> smem[kMaxDevices];        // dynamic shared memory limit set (0: none)
  std::atomic<bool> cluster[kMaxDevices];    // non-portable cluster sizes allowed
};

// Raises `kernel`'s dynamic shared memory limit to `smem` and, when asked,
// allows non-portable cluster sizes, on the current device.
template <typename... KArgs>
inline cudaError_t prepare_kernel(void (*kernel)(KArgs...), size_t smem, bool nonportable_cluster,
                                  KernelAttrs& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool slot = dev >= 0 && dev < kMaxDevices;
  if (!slot || done.smem[dev].load(std::memory_order_acquire) < int(smem)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    if (slot) done.smem[dev].store(int(smem), std::memory_order_release);
  }
  if (nonportable_cluster && (!slot || !done.cluster[dev].load(std::memory_order_acquire))) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    if (slot) done.cluster[dev].store(true, std::memory_order_release);
  }
  return cudaSuccess;
}

// Number of SMs of the current device (read once per device).
inline int device_sms() {
  static std::atomic<int> sms[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (dev >= 0 && dev < kMaxDevices) {
    const int n = sms[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
  }
  int n = 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 152;
  if (dev >= 0 && dev < kMaxDevices) sms[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Launches `kernel` with programmatic stream serialisation (see pdl_wait) and,
// for cluster_x > 1, thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct IdxArgs {
  csa2_dims d;
  int batch;
  const void* idx_k;
  const uint8_t* idx_scales;   // FP4 keys: the scales plane (idx_k + cache rows * 64)
  const int32_t* page_table;
  const int32_t* ctx_len;
  const void* idx_q;
  const float* w;
  const int32_t* pool_in;      // Reindex: pool blocks [B][P]
  const int32_t* pool_len_in;  // Reindex: [B]
  int32_t* pool_out;           // Full: [B][P]
  int32_t* pool_len_out;       // Full: [B]
  int32_t* topk_out;           // [B][K]
  uint8_t* ws;
  WsLayout L;
  float err_coef;              // delta = err_coef * sum_h|w_h|*||q_h||_1 * max|k|
  int early;                   // CSA2_IDX_EARLY_INPUTS: keys, lengths, pages (and the pool) may be read before the wait
};

struct AttnArgs {
  csa2_dims d;
  int batch;
  const uint16_t* q;
  const uint8_t* codes;
  const uint8_t* scales;
  const uint16_t* rope;
  const int32_t* page_table;
  const int32_t* ctx_len;
  const int32_t* topk;
  const uint16_t* swa;
  const int32_t* swa_len;
  float scale;
  float* out;
  float* lse;
  uint8_t* ws;
  WsLayout L;
  int early;                   // Reuse mode: indices and main KV may be read before the wait
  int q_len;                   // queries per sequence (1; 2..4 for a multi-query call, cluster path only)
};

cudaError_t launch_quantize(const uint16_t* x, int64_t n, const int64_t* dst_rows, uint8_t* codes,
                            uint8_t* scales, bool early, cudaStream_t st);
cudaError_t launch_quantize_idx(const uint16_t* x, int64_t n, const int64_t* dst_rows, uint8_t* idx_k,
                                int64_t cache_rows, cudaStream_t st);
cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t n, uint16_t* y,
                              cudaStream_t st);
cudaError_t launch_full(IdxArgs a, cudaStream_t st);
cudaError_t launch_reindex(IdxArgs a, cudaStream_t st);
cudaError_t launch_select(IdxArgs a, bool reindex, cudaStream_t st);
cudaError_t launch_scan_tc(const IdxArgs& a, bool reindex, cudaStream_t st);
cudaError_t launch_scan_fp4(const IdxArgs& a, bool reindex, cudaStream_t st);
cudaError_t launch_attention(AttnArgs a, cudaStream_t st);
size_t select_smem_bytes();
size_t attn_smem_bytes(int heads);

}  // namespace csa2
