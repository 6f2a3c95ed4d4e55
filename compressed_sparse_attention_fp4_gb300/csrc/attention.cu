// attention.cu -- CSA2 sparse MLA-style decode attention (all layer modes).
//
// For one decode query per sequence and every head h, one softmax over the
// entries E = {selected main-KV positions} + {SWA rows} (foosynaptic atlas
// "DeepSeek-V4.1-Flash 梗概", section 3.2, figure "异构 KV": main Q reads
// the Top-K main KV and the exact SWA KV, merged; mode table: Reuse keeps KV
// and indices and changes only Q):
//   key   = [dq(latent) ; rope] (576)  |  SWA row (576)
//   value = dq(latent) (512)           |  SWA row[0:512]
//   out_h = sum_e softmax_e(scale * q_h . key_e) value_e,  lse_h = log-sum-exp.
// FP4 entries are dequantized (exactly, to bf16) just before use (newsaint.id
// "DeepSeek-V4.1-Flash 2026: ...", section 4).
//
// Split-KV: the entry list (K Top-K slots, then W SWA slots) is cut into
// chunks of 64 slots; each CTA computes, for all heads, the chunk's partial
// (max logit m, sum of exp l, unnormalised output o), and a combine kernel
// merges the partials: o = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s.
#include "common.cuh"
#include "kernels.cuh"

namespace csa2 {


constexpr int kKvStride = kDqk + 2;          // bf16 elements per smem row (bank skew)
constexpr int kAttnThreads = 512;

__device__ inline uint32_t e2m1x2_to_f16x2_a(uint32_t byte) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(byte));
  return h2;
}

__device__ inline uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(kAttnThreads) attn_partial_cc_kernel(AttnArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint16_t* kv_s = reinterpret_cast<uint16_t*>(smem_raw);                  // [64][578]
  float* q_s = reinterpret_cast<float*>(smem_raw + kAttnChunk * kKvStride * 2);  // [H][576]
  __shared__ int64_t row_s[kAttnChunk];     // >= 0 main row, -2 - r SWA row r, -1 empty
  __shared__ float p_s[kAttnThreads / 32][kAttnChunk];

  const int b = blockIdx.y, split = blockIdx.x;
  const int H = a.d.heads, K = a.d.topk, W = a.d.swa;
  const bool paged = a.page_table != nullptr;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int64_t n_ctx = checked_ctx(a.ctx_len, a.d, b, paged, a.ws);
  int swl = a.swa_len[b];
  if (swl < 0 || swl > W) {
    if (tid == 0) raise_err(a.ws, CSA2_DEV_SWA_LEN);
    swl = swl < 0 ? 0 : W;
  }
  if (tid < kAttnChunk) {
    int slot = split * kAttnChunk + tid;
    int64_t r = -1;
    if (slot < K) {
      int32_t t = a.topk[int64_t(b) * K + slot];
      if (t >= 0) {
        if (t >= n_ctx) raise_err(a.ws, CSA2_DEV_TOPK_IDX);
        else r = kv_row(a.page_table, a.d, b, t, a.ws);
        if (r < 0) r = -1;
      } else if (t < -1) {
        raise_err(a.ws, CSA2_DEV_TOPK_IDX);
      }
    } else if (slot < K + W && slot - K < swl) {
      r = -2 - (slot - K);
    }
    row_s[tid] = r;
  }
  // query -> fp32 smem
  for (int i = tid; i < H * kDqk; i += blockDim.x)
    q_s[i] = bf16_to_f32(a.q[int64_t(b) * H * kDqk + i]);
  __syncthreads();
  // gather + dequantize the chunk's keys / values into bf16 smem rows
  for (int task = tid; task < kAttnChunk * 36; task += blockDim.x) {
    int e = task / 36, part = task % 36;     // parts 0..31: latent groups, 32..35: rope / tail
    int64_t r = row_s[e];
    uint32_t* dst = reinterpret_cast<uint32_t*>(kv_s + e * kKvStride);
    if (r == -1) {
      if (part < 32) for (int i = 0; i < 8; ++i) dst[part * 8 + i] = 0;
      else for (int i = 0; i < 8; ++i) dst[256 + (part - 32) * 8 + i] = 0;
    } else if (r >= 0) {
      if (part < 32) {
        uint2 c = *reinterpret_cast<const uint2*>(a.codes + r * kCodesPerRow + part * 8);
        uint32_t sc = a.scales[r * kScalesPerRow + part];
        float s = e4m3_to_f32(sc);
        uint32_t cw[2] = {c.x, c.y};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t h2 = e2m1x2_to_f16x2_a((cw[i >> 2] >> (8 * (i & 3))) & 0xFF);
          float lo = __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFF))) * s;
          float hi = __half2float(__ushort_as_half(uint16_t(h2 >> 16))) * s;
          dst[part * 8 + i] = pack_bf16x2(lo, hi);
        }
      } else {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(a.rope + r * kRope) + (part - 32) * 8;
        for (int i = 0; i < 8; ++i) dst[256 + (part - 32) * 8 + i] = src[i];
      }
    } else {
      int sr = int(-2 - r);
      const uint32_t* src = reinterpret_cast<const uint32_t*>(a.swa + (int64_t(b) * W + sr) * kDqk);
      if (part < 32) for (int i = 0; i < 8; ++i) dst[part * 8 + i] = src[part * 8 + i];
      else for (int i = 0; i < 8; ++i) dst[256 + (part - 32) * 8 + i] = src[256 + (part - 32) * 8 + i];
    }
  }
  __syncthreads();
  const int nwarps = blockDim.x / 32;
  float* o_base = reinterpret_cast<float*>(a.ws + a.L.attn_o);
  float* ml_base = reinterpret_cast<float*>(a.ws + a.L.attn_ml);
  for (int h = wid; h < H; h += nwarps) {
    const float* qh = q_s + h * kDqk;
    // logits of entries lane and lane + 32
    float l2[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      int e = lane + 32 * k;
      const uint32_t* kr = reinterpret_cast<const uint32_t*>(kv_s + e * kKvStride);
      float acc = 0.0f;
#pragma unroll 8
      for (int c2 = 0; c2 < kDqk / 2; ++c2) {
        uint32_t kk = kr[c2];
        acc = __fmaf_rn(qh[2 * c2], __uint_as_float(kk << 16), acc);
        acc = __fmaf_rn(qh[2 * c2 + 1], __uint_as_float(kk & 0xFFFF0000u), acc);
      }
      l2[k] = row_s[e] == -1 ? -INFINITY : acc * a.scale;
    }
    float m = fmaxf(l2[0], l2[1]);
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    float p0 = l2[0] == -INFINITY ? 0.0f : expf(l2[0] - m);
    float p1 = l2[1] == -INFINITY ? 0.0f : expf(l2[1] - m);
    float l = p0 + p1;
#pragma unroll
    for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
    p_s[wid][lane] = p0;
    p_s[wid][lane + 32] = p1;
    __syncwarp();
    // output dims [16*lane, 16*lane + 16)
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
    for (int e = 0; e < kAttnChunk; ++e) {
      float p = p_s[wid][e];
      const uint32_t* vr = reinterpret_cast<const uint32_t*>(kv_s + e * kKvStride) + lane * 8;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t vv = vr[i];
        acc[2 * i] = __fmaf_rn(p, __uint_as_float(vv << 16), acc[2 * i]);
        acc[2 * i + 1] = __fmaf_rn(p, __uint_as_float(vv & 0xFFFF0000u), acc[2 * i + 1]);
      }
    }
    __syncwarp();
    int64_t pidx = (int64_t(b) * a.L.splits + split) * H + h;
    float4* op = reinterpret_cast<float4*>(o_base + pidx * kLatent + lane * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) op[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
    if (lane == 0) {
      ml_base[pidx * 2] = m;
      ml_base[pidx * 2 + 1] = l;
    }
  }
}

__global__ void __launch_bounds__(128) attn_combine_kernel(AttnArgs a) {
  const int h = blockIdx.x, b = blockIdx.y, H = a.d.heads, S = a.L.splits;
  const float* o_base = reinterpret_cast<const float*>(a.ws + a.L.attn_o);
  const float* ml = reinterpret_cast<const float*>(a.ws + a.L.attn_ml);
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, ml[((int64_t(b) * S + s) * H + h) * 2]);
  float Lsum = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      int64_t pidx = (int64_t(b) * S + s) * H + h;
      float ms = ml[pidx * 2], ls = ml[pidx * 2 + 1];
      if (ms == -INFINITY) continue;
      float wgt = expf(ms - M);
      Lsum += wgt * ls;
      float4 o = reinterpret_cast<const float4*>(o_base + pidx * kLatent)[threadIdx.x];
      acc.x += wgt * o.x; acc.y += wgt * o.y; acc.z += wgt * o.z; acc.w += wgt * o.w;
    }
  }
  float inv = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
  float4 r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  reinterpret_cast<float4*>(a.out + (int64_t(b) * H + h) * kLatent)[threadIdx.x] = r;
  if (threadIdx.x == 0) a.lse[int64_t(b) * H + h] = (Lsum > 0.0f) ? M + logf(Lsum) : -INFINITY;
}

size_t attn_smem_bytes(int heads) {
  return size_t(kAttnChunk) * kKvStride * 2 + size_t(heads) * kDqk * 4;
}

cudaError_t launch_attention(AttnArgs a, cudaStream_t st) {
  size_t smem = attn_smem_bytes(a.d.heads);
  cudaError_t e = cudaFuncSetAttribute(attn_partial_cc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  attn_partial_cc_kernel<<<dim3(unsigned(a.L.splits), unsigned(a.batch)), kAttnThreads, smem, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_combine_kernel<<<dim3(unsigned(a.d.heads), unsigned(a.batch)), 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace csa2
