// indexer.cu -- CSA2 hierarchical sparse indexer (Full scan, pool, Top-K,
// Reindex).
//
// What it computes (foosynaptic atlas "DeepSeek-V4.1-Flash 梗概", section
// 3.2, "Hierarchical Sparse Indexer (decoder)": the first Full layer builds a
// pool of Top-2048 blocks of 8, later Reindex layers score only inside the
// pool and take Top-512; newsaint.id "DeepSeek-V4.1-Flash 2026: ...", section
// 3 and HierarchicalSparseIndexer in section 8):
//   s_t  = sum_h w_h * ReLU(q_h . k_t)      (weighted multi-head indexer score)
//   bs_j = max_{t in block j} s_t           (block of 8 positions)
//   pool = Top-P blocks, Top-K = Top-K pool positions, ties to the lower index.
//
// The ranking is defined on exact scores (head dots rounded once to fp64,
// head sum in fp64).  The scan computes fast approximate scores v with a
// rigorous bound |v - s| <= delta (per block of 8).  Selecting the P best
// out of n items then only needs exact scores for the "band": with
// mu = P-th largest of (v + delta) and lambda = P-th largest of (v - delta),
//   v - delta > mu                 -> certainly selected,
//   v + delta < lambda             -> certainly not selected,
//   otherwise                      -> re-scored exactly, then ranked.
// (The true P-th best score lies in [lambda, mu].)  The result equals the
// selection made on exact scores.
#include <cmath>

#include "common.cuh"
#include "kernels.cuh"
#include "profile.cuh"

namespace csa2 {


// ===========================================================================
// Approximate scan on CUDA cores (fp32 FMA).  One thread per position, 256
// positions per CTA (32 blocks of 8 = one warp-octet per block).
// Full mode: positions [256*tile, 256*tile + 256) of sequence blockIdx.y.
// Reindex mode: items [256*tile, ...) of the pool, item i = position
// 8*pool[i/8] + i%8.
// ===========================================================================
template <bool kFp8, int kDi>
__global__ void __launch_bounds__(256) scan_cc_kernel(IdxArgs a, bool reindex) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float q_s[kDi][kMaxIdxHeads];     // [c][h]
  __shared__ float w_s[kMaxIdxHeads];
  __shared__ float wq_s;
  const int b = blockIdx.y;
  const int hi = a.d.idx_heads;
  const bool paged = a.page_table != nullptr;
  const int64_t n_ctx = checked_ctx(a.ctx_len, a.d, b, paged, a.ws);

  for (int i = threadIdx.x; i < kDi * kMaxIdxHeads; i += blockDim.x) {
    int c = i / kMaxIdxHeads, h = i % kMaxIdxHeads;
    float v = 0.0f;
    if (h < hi) {
      int64_t qi = (int64_t(b) * hi + h) * kDi + c;
      v = kFp8 ? bf16_to_f32(reinterpret_cast<const uint16_t*>(a.idx_q)[qi])
               : reinterpret_cast<const float*>(a.idx_q)[qi];
    }
    q_s[c][h] = v;
  }
  if (threadIdx.x < kMaxIdxHeads)
    w_s[threadIdx.x] = threadIdx.x < hi ? a.w[int64_t(b) * hi + threadIdx.x] : 0.0f;
  __syncthreads();
  if (threadIdx.x < 32) {
    // sum_h |w_h| * ||q_h||_1, rounded upwards (an upper bound).
    float acc = 0.0f;
    for (int h = 0; h < hi; ++h) {
      float l1 = 0.0f;
      for (int c = threadIdx.x; c < kDi; c += 32) l1 = __fadd_ru(l1, fabsf(q_s[c][h]));
      for (int o = 16; o; o >>= 1) l1 = __fadd_ru(l1, __shfl_xor_sync(0xFFFFFFFFu, l1, o));
      acc = __fadd_ru(acc, __fmul_ru(fabsf(w_s[h]), l1));
    }
    if (threadIdx.x == 0) wq_s = acc;
  }
  __syncthreads();

  const int64_t item = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  int64_t t = item;
  bool valid;
  int64_t P8 = int64_t(a.d.pool_blocks) * kBlock;
  if (!reindex) {
    valid = item < n_ctx;
  } else {
    int32_t plen = a.pool_len_in[b];
    int64_t j = item >> 3;
    valid = item < P8 && j < plen && plen <= a.d.pool_blocks;
    if (plen > a.d.pool_blocks || plen < 0) raise_err(a.ws, CSA2_DEV_POOL);
    if (valid) {
      int32_t blk = a.pool_in[int64_t(b) * a.d.pool_blocks + j];
      if (blk < 0 || int64_t(blk) * kBlock >= n_ctx) {
        raise_err(a.ws, CSA2_DEV_POOL);
        valid = false;
      }
      t = int64_t(blk) * kBlock + (item & 7);
      valid = valid && t < n_ctx;
    }
  }
  float acc[kMaxIdxHeads];
#pragma unroll
  for (int h = 0; h < kMaxIdxHeads; ++h) acc[h] = 0.0f;
  float kmax = 0.0f;
  int64_t row = valid ? kv_row(a.page_table, a.d, b, t, a.ws) : -1;
  valid = valid && row >= 0;
  if (valid) {
    if (kFp8) {
      const uint4* kp = reinterpret_cast<const uint4*>(
          reinterpret_cast<const uint8_t*>(a.idx_k) + row * kDi);
#pragma unroll 1
      for (int ch = 0; ch < kDi / 16; ++ch) {
        uint4 v = __ldg(kp + ch);
        uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            uint32_t h2 = e4m3x2_to_f16x2(uint16_t(wv[i] >> (16 * p)));
            float k0 = __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFF)));
            float k1 = __half2float(__ushort_as_half(uint16_t(h2 >> 16)));
            int c = ch * 16 + i * 4 + p * 2;
            kmax = fmaxf(kmax, fmaxf(fabsf(k0), fabsf(k1)));
#pragma unroll
            for (int h = 0; h < kMaxIdxHeads; ++h) {
              acc[h] = __fmaf_rn(q_s[c][h], k0, acc[h]);
              acc[h] = __fmaf_rn(q_s[c + 1][h], k1, acc[h]);
            }
          }
        }
      }
    } else {
      const float4* kp = reinterpret_cast<const float4*>(
          reinterpret_cast<const float*>(a.idx_k) + row * kDi);
#pragma unroll 1
      for (int ch = 0; ch < kDi / 4; ++ch) {
        float4 v = __ldg(kp + ch);
        float kv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          int c = ch * 4 + i;
          kmax = fmaxf(kmax, fabsf(kv[i]));
#pragma unroll
          for (int h = 0; h < kMaxIdxHeads; ++h) acc[h] = __fmaf_rn(q_s[c][h], kv[i], acc[h]);
        }
      }
    }
  }
  float s = 0.0f;
#pragma unroll
  for (int h = 0; h < kMaxIdxHeads; ++h) s = __fmaf_rn(w_s[h], fmaxf(acc[h], 0.0f), s);
  if (!valid) s = -INFINITY;
  // block of 8 = 8 consecutive lanes
  float bmax = s, bk = kmax;
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    bmax = fmaxf(bmax, __shfl_xor_sync(0xFFFFFFFFu, bmax, o));
    bk = fmaxf(bk, __shfl_xor_sync(0xFFFFFFFFu, bk, o));
  }
  float delta = __fmul_ru(__fmul_ru(a.err_coef, wq_s), bk);
  float* ws_f = reinterpret_cast<float*>(a.ws);
  if (!reindex) {
    if (valid) ws_f[(a.L.pos_scores >> 2) + int64_t(b) * a.d.max_ctx + t] = s;
    int64_t j = item >> 3;
    if ((threadIdx.x & 7) == 0 && j * kBlock < n_ctx) {
      ws_f[(a.L.blk_scores >> 2) + int64_t(b) * a.L.nb_max + j] = bmax;
      ws_f[(a.L.blk_delta >> 2) + int64_t(b) * a.L.nb_max + j] = delta;
    }
  } else if (item < P8) {
    ws_f[(a.L.ri_scores >> 2) + int64_t(b) * P8 + item] = s;
    if ((threadIdx.x & 7) == 0) ws_f[(a.L.ri_delta >> 2) + int64_t(b) * a.d.pool_blocks + (item >> 3)] = delta;
  }
}

// ===========================================================================
// Host-side launchers
// ===========================================================================
static double gamma_n(int n, double u) { return n * u / (1.0 - n * u); }

// Bound constant of the CUDA-core scan: per-head fp32 FMA chains of Di terms,
// the fp32 FMA head sum of Hi terms, and the fp64 rounding of the exact
// score, all relative to sum_h |w_h| * sum_c |q_hc k_tc|.
static float cc_err_coef(int di, int hi) {
  const double u32 = std::ldexp(1.0, -24), u64 = std::ldexp(1.0, -53);
  double gd = gamma_n(di, u32), gh = gamma_n(hi + 1, u32), g64 = gamma_n(hi + 2, u64);
  double c = (gd + gh * (1.0 + gd) + g64) * 1.01;
  return float(c * (1.0 + 1e-6));
}

cudaError_t launch_full(IdxArgs a, cudaStream_t st) {
  const bool fp8 = a.d.idx_k_dtype == CSA2_IDXK_E4M3;
  a.err_coef = cc_err_coef(a.d.idx_dim, a.d.idx_heads);
  cudaError_t e;
  if (fp8) {
    // E4M3 keys: tensor-core scan (tcgen05), bound from the |A| . |q| product
    e = launch_scan_tc(a, false, st);
  } else if (a.d.idx_k_dtype == CSA2_IDXK_FP4) {
    // FP4 keys: exact group dots on the tensor cores, scales in fp32
    e = launch_scan_fp4(a, false, st);
  } else {
    dim3 grid(unsigned((a.d.max_ctx + 255) / 256), unsigned(a.batch));
    CSA2_PROFILED(st, "indexer_scan_cuda_core",
                  (e = launch_pdl(scan_cc_kernel<false, 64>, grid, dim3(256), 0, st, 1, a, false)));
  }
  if (e != cudaSuccess) return e;
  return launch_select(a, false, st);
}

cudaError_t launch_reindex(IdxArgs a, cudaStream_t st) {
  const bool fp8 = a.d.idx_k_dtype == CSA2_IDXK_E4M3;
  a.err_coef = cc_err_coef(a.d.idx_dim, a.d.idx_heads);
  int64_t P8 = int64_t(a.d.pool_blocks) * kBlock;
  dim3 grid(unsigned((P8 + 255) / 256), unsigned(a.batch));
  cudaError_t e;
  if (fp8) {
    e = launch_scan_tc(a, true, st);
  } else if (a.d.idx_k_dtype == CSA2_IDXK_FP4) {
    e = launch_scan_fp4(a, true, st);
  } else {
    CSA2_PROFILED(st, "reindex_score_cuda_core",
                  (e = launch_pdl(scan_cc_kernel<false, 64>, grid, dim3(256), 0, st, 1, a, true)));
  }
  if (e != cudaSuccess) return e;
  return launch_select(a, true, st);
}

}  // namespace csa2
