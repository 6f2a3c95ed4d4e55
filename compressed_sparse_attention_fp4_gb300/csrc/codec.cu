// codec.cu -- FP4 main-KV codec: bf16 latent <-> packed E2M1 + E4M3 scales.
//
// Format (foosynaptic atlas "DeepSeek-V4.1-Flash 梗概", section 3.2, "FP4 main
// KV": E2M1 with one E4M3 scale per 16 channels; newsaint.id "DeepSeek-V4.1-
// Flash 2026: ...", section 8, FP4Quantizer: levels {0,.5,1,1.5,2,3,4,6},
// scale = amax/6 limited to 448, no second-level scale).
//
// Rounding: the reading fp4.cuh states and implements (shared with the
// FP4 indexer keys and query).
//
// Layout: one warp per 512-channel row.  Round r in {0,1} covers channels
// [256r, 256r+256): lane l loads 8 bf16 (16 B, coalesced), lanes 2g and 2g+1
// share group g, and each lane stores 4 packed bytes (coalesced 128 B per
// warp) and, for even lanes, one scale byte.
#include "common.cuh"
#include "fp4.cuh"
#include "kernels.cuh"
#include "profile.cuh"

namespace csa2 {

__global__ void __launch_bounds__(256) quantize_kernel(const uint4* __restrict__ x, int64_t n,
                                                       const int64_t* __restrict__ dst_rows,
                                                       uint32_t* __restrict__ codes,
                                                       uint8_t* __restrict__ scales, int early) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  // early inputs: the kernel before writes none of x / dst_rows and touches
  // none of the destination rows; the rows are written while it runs, and
  // this grid completes only after it (the wait at the end), so whatever
  // waits on this grid also sees that kernel's results
  if (!early) pdl_wait();
  pdl_launch_dependents();
  for (int64_t row = warp; row < n; row += nwarps) {
    int64_t dst = dst_rows ? dst_rows[row] : row;
    if (dst < 0) continue;
    uint4 v[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) v[r] = __ldcs(x + row * 64 + r * 32 + lane);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      uint32_t sc;
      const uint32_t packed = fp4_quantize_half_group(v[r], &sc);
      codes[dst * 64 + r * 32 + lane] = packed;
      if ((lane & 1) == 0) scales[dst * 32 + r * 16 + (lane >> 1)] = uint8_t(sc);
    }
  }
  if (early) pdl_wait();
}

// Two E2M1 nibbles (low nibble = first) -> f16x2 (low half = first), exact.
__device__ inline uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(byte));
  return h2;
}

__device__ inline uint32_t f16x2_to_bf16x2(uint32_t h2) {
  float lo = __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFF)));
  float hi = __half2float(__ushort_as_half(uint16_t(h2 >> 16)));
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(256) dequantize_kernel(const uint2* __restrict__ codes,
                                                         const uint8_t* __restrict__ scales,
                                                         int64_t n, uint4* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  pdl_wait();
  pdl_launch_dependents();
  for (int64_t row = warp; row < n; row += nwarps) {
    uint2 c = __ldcs(codes + row * 32 + lane);          // 16 nibbles = group `lane`
    uint32_t sc = scales[row * 32 + lane];
    uint32_t s2 = e4m3x2_to_f16x2(uint16_t(sc | (sc << 8)));
    __half2 sh = *reinterpret_cast<__half2*>(&s2);
    uint32_t cw[2] = {c.x, c.y};
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t byte = (cw[i >> 2] >> (8 * (i & 3))) & 0xFF;
      uint32_t h2 = e2m1x2_to_f16x2(byte);
      __half2 v = __hmul2(*reinterpret_cast<__half2*>(&h2), sh);   // exact
      out[i] = f16x2_to_bf16x2(*reinterpret_cast<uint32_t*>(&v));
    }
    __stcs(y + row * 64 + lane * 2, make_uint4(out[0], out[1], out[2], out[3]));
    __stcs(y + row * 64 + lane * 2 + 1, make_uint4(out[4], out[5], out[6], out[7]));
  }
}

// FP4 indexer keys: rows of 128 bf16 channels into the two-plane indexer-K
// cache (codes [rows][64], then scales [rows][8]).  A warp takes two rows:
// lane l covers row 2w + l/16, channels 8 (l % 16) .. + 7 (16 B of input, 4
// bytes of codes); lanes 2g and 2g+1 of a half-warp share group g.  Rows whose
// destination is negative or not below cache_rows are skipped.
__global__ void __launch_bounds__(256) quantize_idx_kernel(const uint4* __restrict__ x, int64_t n,
                                                           const int64_t* __restrict__ dst_rows,
                                                           uint32_t* __restrict__ codes,
                                                           uint8_t* __restrict__ scales, int64_t cache_rows) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  pdl_wait();
  pdl_launch_dependents();
  const int half = lane >> 4, part = lane & 15;
  for (int64_t pair = warp; 2 * pair < n; pair += nwarps) {
    const int64_t row = 2 * pair + half;
    const bool have = row < n;
    const int64_t dst = have ? (dst_rows ? dst_rows[row] : row) : -1;
    const uint4 v = have ? __ldcs(x + row * 16 + part) : make_uint4(0, 0, 0, 0);
    uint32_t sc;
    const uint32_t packed = fp4_quantize_half_group(v, &sc);   // all 32 lanes take part
    if (dst >= 0 && dst < cache_rows) {
      codes[dst * 16 + part] = packed;
      if ((part & 1) == 0) scales[dst * 8 + (part >> 1)] = uint8_t(sc);
    }
  }
}

static int codec_grid(int64_t n) {
  const int sms = device_sms();
  int64_t want = (n + 7) / 8;                    // 8 warps per block, 1 row per warp
  int64_t cap = int64_t(sms) * 8;                // 8 blocks of 256 per SM, grid-stride
  return int(want < cap ? (want > 0 ? want : 1) : cap);
}

cudaError_t launch_quantize(const uint16_t* x, int64_t n, const int64_t* dst_rows, uint8_t* codes,
                            uint8_t* scales, bool early, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  cudaError_t e;
  CSA2_PROFILED(st, "fp4_quantize",
                (e = launch_pdl(quantize_kernel, dim3(codec_grid(n)), dim3(256), 0, st, 1,
                                reinterpret_cast<const uint4*>(x), n, dst_rows,
                                reinterpret_cast<uint32_t*>(codes), scales, early ? 1 : 0)));
  return e;
}

cudaError_t launch_quantize_idx(const uint16_t* x, int64_t n, const int64_t* dst_rows, uint8_t* idx_k,
                                int64_t cache_rows, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  cudaError_t e;
  CSA2_PROFILED(st, "fp4_idx_quantize",
                (e = launch_pdl(quantize_idx_kernel, dim3(codec_grid((n + 1) / 2)), dim3(256), 0, st, 1,
                                reinterpret_cast<const uint4*>(x), n, dst_rows,
                                reinterpret_cast<uint32_t*>(idx_k), idx_k + cache_rows * 64, cache_rows)));
  return e;
}

cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t n, uint16_t* y,
                              cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  cudaError_t e;
  CSA2_PROFILED(st, "fp4_dequantize",
                (e = launch_pdl(dequantize_kernel, dim3(codec_grid(n)), dim3(256), 0, st, 1,
                                reinterpret_cast<const uint2*>(codes), scales, n, reinterpret_cast<uint4*>(y))));
  return e;
}

}  // namespace csa2
