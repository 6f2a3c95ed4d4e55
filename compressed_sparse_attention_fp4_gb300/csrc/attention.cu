// attention.cu -- CSA2 sparse MLA-style decode attention (all layer modes) on
// the tcgen05 tensor cores.
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
// chunks of 128 slots.  For each chunk:
//   1. its 128 entries are gathered and dequantized from FP4 to bf16 into
//      shared memory (128-byte swizzled, one 16 KB region per 64 channels);
//      the query [64 heads x 576] and a window that starts a chunk come by TMA;
//   2. S^T[128 entries x 64 heads] = KV . Q^T on tcgen05 (M=128, N=64, bf16 in,
//      fp32 in tensor memory);
//   3. softmax over the entries (= TMEM lanes): per-head max and sum by
//      butterfly reduce-scatter and across the 4 lane quarters; P^T is written
//      back as bf16 hi + lo parts, so its rounding stays near 2^-17;
//   4. O^T = V^T . P^T on tcgen05 (the same KV tile read MN-major), M-tiles of
//      128 dims, hi and lo accumulated together;
//   5. the chunks of the sequence are merged: o = sum_s 2^(m_s - M) o_s / L,
//      L = sum_s 2^(m_s - M) l_s, lse = M ln 2 + ln L (m in base-2 logits).
//
// attn_pair_kernel (at most 8 chunks, the usual case): two CTAs per chunk
// split the 576 channels (latent 0..255 | latent 256..511 + rope), exchange
// their S^T partials through shared memory and each computes O^T for its 256
// value dimensions.  The 2 x chunks CTAs of a sequence form one thread-block
// cluster: every chunk copies its per-head (m_s, l_s) into every CTA's shared
// memory, on an mbarrier that counts the bytes; the chunk that finishes first
// (the TMA-loaded SWA window) zeroes the output early and signals the other
// chunks of its half; each CTA then forms M and L, scales its O^T part and
// adds it into the output with coalesced reduce-adds (red.global.add.f32)
// straight from tensor memory.  The order of the additions is not fixed, so
// the last bits of the output may differ between runs.
//
// attn_partial_tc_kernel + attn_combine_kernel (more chunks): one CTA per
// chunk writes its unnormalised O_s and (m_s, l_s) (natural-log m) to the
// workspace and the combine kernel merges them.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"
#include "profile.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace cg = cooperative_groups;

namespace csa2 {

constexpr int kAttnThreads = 512;
constexpr int kEntries = 128;                       // entries per CTA (= MMA M)
constexpr int kQRows = 64;                          // MMA N (heads, zero padded)
constexpr int kRegion = kEntries * 128;             // 64 channels x 128 entries, bytes
constexpr int kQRegion = kQRows * 128;
constexpr int kKvBytes = 9 * kRegion;               // 576 channels
constexpr int kQBytes = 9 * kQRegion;
constexpr uint32_t kTmemCols = 512;                 // S^T: 64 cols, O^T: 4 x 64 cols

static_assert(kEntries == kAttnChunk, "split size of the workspace layout");

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

// Reduces 16 values per lane over the warp's 32 lanes by a butterfly
// reduce-scatter (8 + 4 + 2 + 1 + 1 shuffles instead of 16 x 5): returns the
// reduction of value index butterfly_index(lane), held by lanes 2i and 2i+1.
__device__ inline int butterfly_index(int lane) {
  return (((lane >> 4) & 1) << 3) | (((lane >> 3) & 1) << 2) | (((lane >> 2) & 1) << 1) | ((lane >> 1) & 1);
}

template <bool kMax>
__device__ inline float butterfly16(const float (&v)[16], int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float y[8], z[4], w[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float keep = b4 ? v[8 + i] : v[i], give = b4 ? v[i] : v[8 + i];
    y[i] = op(keep, __shfl_xor_sync(0xFFFFFFFFu, give, 16));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b3 ? y[4 + i] : y[i], give = b3 ? y[i] : y[4 + i];
    z[i] = op(keep, __shfl_xor_sync(0xFFFFFFFFu, give, 8));
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b2 ? z[2 + i] : z[i], give = b2 ? z[i] : z[2 + i];
    w[i] = op(keep, __shfl_xor_sync(0xFFFFFFFFu, give, 4));
  }
  const float keep = b1 ? w[1] : w[0], give = b1 ? w[0] : w[1];
  float u = op(keep, __shfl_xor_sync(0xFFFFFFFFu, give, 2));
  return op(u, __shfl_xor_sync(0xFFFFFFFFu, u, 1));
}

__device__ inline void st_shared_v4(uint8_t* base, uint32_t off, uint4 v) {
  *reinterpret_cast<uint4*>(base + off) = v;
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_partial_tc_kernel(AttnArgs a, const __grid_constant__ CUtensorMap qmap,
                           const __grid_constant__ CUtensorMap swamap, int swa_tma_split) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte swizzled operands need 1024-byte aligned regions
  uint8_t* kv_s = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);   // 9 x 16 KB
  uint8_t* q_s = kv_s + kKvBytes;                   // 9 regions x 8 KB; later P^T hi / lo
  __shared__ uint64_t bar_ld, bar_s, bar_o;
  __shared__ uint32_t tmem_slot;
  __shared__ int64_t row_s[kEntries];               // >= 0 main row, -2 - r SWA row r, -1 empty
  __shared__ __align__(16) float red_m[4][4][16];
  __shared__ __align__(16) float red_l[4][4][16];

  const int b = blockIdx.y, split = blockIdx.x;
  const int H = a.d.heads, K = a.d.topk, W = a.d.swa;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // set-up that touches no global memory, then wait for the previous kernel
  if (wid == 0) tc::tmem_alloc(&tmem_slot, kTmemCols);
  if (tid == 0) {
    tc::mbar_init(&bar_ld, 1);
    tc::mbar_init(&bar_s, 1);
    tc::mbar_init(&bar_o, 1);
    tc::fence_mbar_init();
  }
  pdl_wait();
  pdl_launch_dependents();
  const bool paged = a.page_table != nullptr;
  const bool swa_tma = split == swa_tma_split;      // this CTA's rows are the SWA window
  const int64_t n_ctx = checked_ctx(a.ctx_len, a.d, b, paged, a.ws);
  int swl = a.swa_len[b];
  if (swl < 0 || swl > W) {
    if (tid == 0) raise_err(a.ws, CSA2_DEV_SWA_LEN);
    swl = swl < 0 ? 0 : W;
  }
  if (tid < kEntries) {
    int slot = split * kEntries + tid;
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
  tc::tc_fence_before_sync();
  __syncthreads();
  tc::tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;

  // ---- TMA: the query (9 boxes of 64 channels x 64 heads) and, for the
  //      window's CTA, the SWA rows (9 boxes of 64 channels x 128 rows) ----------
  if (tid == 0) {
    tc::mbar_expect_tx(&bar_ld, uint32_t(kQBytes) + (swa_tma ? uint32_t(kKvBytes) : 0u));
    for (int kb = 0; kb < 9; ++kb) tc::tma_load_2d(&qmap, q_s + kb * kQRegion, 64 * kb, b * H, &bar_ld);
    if (swa_tma)
      for (int kb = 0; kb < 9; ++kb) tc::tma_load_2d(&swamap, kv_s + kb * kRegion, 64 * kb, b * W, &bar_ld);
  }
  // ---- FP4 entries: gather (all loads first), dequantize to bf16 -------------------
  if (!swa_tma) {
    // latent: task = (entry, pair of 16-channel groups); 4 tasks per thread
    uint4 cd[4];
    uint32_t sc[4];
    int64_t rr[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int task = tid + k * kAttnThreads, e = task >> 4, gp = task & 15;
      rr[k] = row_s[e];
      cd[k] = make_uint4(0, 0, 0, 0);
      sc[k] = 0;
      if (rr[k] >= 0) {
        cd[k] = __ldg(reinterpret_cast<const uint4*>(a.codes + rr[k] * kCodesPerRow) + gp);
        sc[k] = __ldg(reinterpret_cast<const uint16_t*>(a.scales + rr[k] * kScalesPerRow) + gp);
      }
    }
    // rope: task = (entry, 16-byte chunk); 2 tasks per thread
    uint4 rp[2];
    int64_t rr2[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int task = tid + k * kAttnThreads, e = task >> 3, rc = task & 7;
      rr2[k] = row_s[e];
      rp[k] = make_uint4(0, 0, 0, 0);
      if (rr2[k] >= 0) rp[k] = __ldg(reinterpret_cast<const uint4*>(a.rope + rr2[k] * kRope) + rc);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int task = tid + k * kAttnThreads, e = task >> 4, gp = task & 15;
      if (rr[k] <= -2) continue;                     // SWA row: copied below
      uint32_t cw[4] = {cd[k].x, cd[k].y, cd[k].z, cd[k].w};
#pragma unroll
      for (int g = 0; g < 2; ++g) {                  // two 16-channel groups
        float s = e4m3_to_f32((sc[k] >> (8 * g)) & 0xFF);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t h2 = e2m1x2_to_f16x2_a((cw[2 * g + (i >> 2)] >> (8 * (i & 3))) & 0xFF);
          float lo = __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFF))) * s;
          float hi = __half2float(__ushort_as_half(uint16_t(h2 >> 16))) * s;
          w[i] = pack_bf16x2(lo, hi);
        }
        const int part = 2 * gp + g;                 // 16-channel group index 0..31
        const uint32_t region = part >> 2, ch0 = (part & 3) * 2;
        st_shared_v4(kv_s, region * kRegion + tc::sw128_offset(e, ch0), make_uint4(w[0], w[1], w[2], w[3]));
        st_shared_v4(kv_s, region * kRegion + tc::sw128_offset(e, ch0 + 1), make_uint4(w[4], w[5], w[6], w[7]));
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int task = tid + k * kAttnThreads, e = task >> 3, rc = task & 7;
      if (rr2[k] <= -2) continue;
      st_shared_v4(kv_s, 8 * kRegion + tc::sw128_offset(e, rc), rp[k]);
    }
    // SWA rows of a CTA the window does not start on a 128-row boundary for
#pragma unroll 4
    for (int task = tid; task < kEntries * 72; task += kAttnThreads) {
      const int e = task / 72, c = task % 72;
      const int64_t r = row_s[e];
      if (r > -2) continue;
      uint4 v = __ldg(reinterpret_cast<const uint4*>(a.swa + (int64_t(b) * W + (-2 - r)) * kDqk) + c);
      st_shared_v4(kv_s, (c >> 3) * kRegion + tc::sw128_offset(e, c & 7), v);
    }
  }
  bool ok = tc::mbar_wait_bounded(&bar_ld, 0);
  if (swa_tma) {
    // window rows past swa_len (or past W) are not entries: zero them so that
    // P = 0 never meets a non-finite value
    for (int task = tid; task < kEntries * 72; task += kAttnThreads) {
      const int e = task / 72, c = task % 72;
      if (row_s[e] == -1) st_shared_v4(kv_s, (c >> 3) * kRegion + tc::sw128_offset(e, c & 7), make_uint4(0, 0, 0, 0));
    }
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before_sync();
  __syncthreads();

  // ---- S^T = KV . Q^T ------------------------------------------------------------
  const uint32_t kv_addr = tc::smem_u32(kv_s), q_addr = tc::smem_u32(q_s);
  if (tid == 0) {
    tc::tc_fence_after_sync();
    constexpr uint32_t idS = tc::idesc_bf16(kEntries, kQRows, 0, 0);
    // descriptors are formed once; an offset of x bytes adds x/16 to the
    // start-address field (the operands lie below 256 KB, so it never carries)
    const uint64_t ad0 = tc::smem_desc(kv_addr, 16, 1024, 2), bd0 = tc::smem_desc(q_addr, 16, 1024, 2);
#pragma unroll
    for (int ks = 0; ks < 36; ++ks) {
      const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
      tc::mma_bf16(tmem, ad0 + ((kb * kRegion + off) >> 4), bd0 + ((kb * kQRegion + off) >> 4), idS, ks > 0);
    }
    tc::mma_commit(&bar_s);
  }
  ok = tc::mbar_wait_bounded(&bar_s, 0) && ok;
  tc::tc_fence_after_sync();

  // ---- softmax over the 128 entries (TMEM lanes) ------------------------------
  const int quarter = wid & 3, hg = wid >> 2;       // lanes 32*quarter.., heads 16*hg..
  const int e = quarter * 32 + lane;
  const bool valid = row_s[e] != -1;
  float x[16];
  tc::tmem_ld16(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(hg * 16), x);
  const float c2 = a.scale * 1.4426950408889634f;   // logits in base 2
#pragma unroll
  for (int j = 0; j < 16; ++j) x[j] = valid ? x[j] * c2 : -INFINITY;
  {
    const float m = butterfly16<true>(x, lane);
    if ((lane & 1) == 0) red_m[hg][quarter][butterfly_index(lane)] = m;
  }
  __syncthreads();
  float p[16];
#pragma unroll
  for (int j4 = 0; j4 < 4; ++j4) {
    float4 m4[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) m4[q] = reinterpret_cast<const float4*>(&red_m[hg][q][0])[j4];
    const float Mj[4] = {fmaxf(fmaxf(m4[0].x, m4[1].x), fmaxf(m4[2].x, m4[3].x)),
                         fmaxf(fmaxf(m4[0].y, m4[1].y), fmaxf(m4[2].y, m4[3].y)),
                         fmaxf(fmaxf(m4[0].z, m4[1].z), fmaxf(m4[2].z, m4[3].z)),
                         fmaxf(fmaxf(m4[0].w, m4[1].w), fmaxf(m4[2].w, m4[3].w))};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = 4 * j4 + i;
      p[j] = (Mj[i] == -INFINITY || x[j] == -INFINITY) ? 0.0f : exp2f(x[j] - Mj[i]);
    }
  }
  {
    const float l = butterfly16<false>(p, lane);
    if ((lane & 1) == 0) red_l[hg][quarter][butterfly_index(lane)] = l;
  }
  // P^T rows (entry e): heads 16*hg.. as 2 chunks, hi and lo bf16 parts.
  // The query buffer is free: the S^T MMAs completed (bar_s) before this.
  uint8_t* p_hi = q_s;
  uint8_t* p_lo = q_s + kRegion;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    uint32_t wh[4], wl[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float v0 = p[8 * t + 2 * i], v1 = p[8 * t + 2 * i + 1];
      uint32_t hb = pack_bf16x2(v0, v1);
      float h0 = __uint_as_float(hb << 16), h1 = __uint_as_float(hb & 0xFFFF0000u);
      wh[i] = hb;
      wl[i] = pack_bf16x2(v0 - h0, v1 - h1);
    }
    uint32_t off = tc::sw128_offset(e, hg * 2 + t);
    st_shared_v4(p_hi, off, make_uint4(wh[0], wh[1], wh[2], wh[3]));
    st_shared_v4(p_lo, off, make_uint4(wl[0], wl[1], wl[2], wl[3]));
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before_sync();
  __syncthreads();
  float* ml_base = reinterpret_cast<float*>(a.ws + a.L.attn_ml);
  const int64_t prow = (int64_t(b) * a.L.splits + split) * H;
  if (quarter == 0 && lane < 16) {
    int h = hg * 16 + lane;
    if (h < H) {
      float M = fmaxf(fmaxf(red_m[hg][0][lane], red_m[hg][1][lane]), fmaxf(red_m[hg][2][lane], red_m[hg][3][lane]));
      float L = red_l[hg][0][lane] + red_l[hg][1][lane] + red_l[hg][2][lane] + red_l[hg][3][lane];
        ml_base[(prow + h) * 2] = M == -INFINITY ? -INFINITY : M * 0.6931471805599453f;
        ml_base[(prow + h) * 2 + 1] = L;
    }
  }

  // ---- O^T = V^T . P^T  (4 M-tiles of 128 channels; hi and lo parts) -------------
  if (tid == 0) {
    tc::tc_fence_after_sync();
    constexpr uint32_t idO = tc::idesc_bf16(kEntries, kQRows, 1, 1);
    const uint64_t av0 = tc::smem_desc(kv_addr, kRegion, 1024, 2);
    const uint64_t bp0[2] = {tc::smem_desc(tc::smem_u32(p_hi), kRegion, 1024, 2),
                             tc::smem_desc(tc::smem_u32(p_lo), kRegion, 1024, 2)};
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
      for (int part = 0; part < 2; ++part) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc::mma_bf16(tmem + 64 + 64 * mt, av0 + (((2 * mt) * kRegion + ks * 2048) >> 4),
                       bp0[part] + ((ks * 2048) >> 4), idO, part > 0 || ks > 0);
      }
    }
    tc::mma_commit(&bar_o);
  }
  ok = tc::mbar_wait_bounded(&bar_o, 0) && ok;
  tc::tc_fence_after_sync();
  if (!ok && tid == 0) raise_err(a.ws, CSA2_DEV_TIMEOUT);

  // ---- O^T through shared memory as [head][dim] (the KV tile is no longer
  //      read: the PV MMAs completed), then one bulk copy of 2 KB per head
  //      into the workspace partials that the combine kernel merges --------
  float* obuf = reinterpret_cast<float*>(kv_s);
#pragma unroll 1
  for (int mt = 0; mt < 4; ++mt) {
    float o[16];
    tc::tmem_ld16(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(64 + 64 * mt + hg * 16), o);
    const int dim = mt * 128 + quarter * 32 + lane;
#pragma unroll
    for (int j = 0; j < 16; ++j) obuf[(hg * 16 + j) * kLatent + dim] = o[j];
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before_sync();
  __syncthreads();
  if (wid == 0) tc::tmem_dealloc(tmem, kTmemCols);
  if (tid < H) {
    const uint32_t src = tc::smem_u32(obuf + tid * kLatent);
    float* dst = reinterpret_cast<float*>(a.ws + a.L.attn_o) + (prow + tid) * kLatent;
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(dst), "r"(src), "r"(uint32_t(kLatent * 4))
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");   // shared source read out
  }
}

// ---------------------------------------------------------------------------
// Channel-split pairs.  Every 128-entry chunk is served by two CTAs: half 0
// takes latent channels 0..255, half 1 latent channels 256..511 and the rope
// (64).  Each gathers, dequantizes and multiplies only its channels
// (S^T partial, M=128, N=64, K=256 or 320), the pair exchanges the partial
// S^T through shared memory (one bulk copy into the partner, completing on
// its mbarrier), both
// form the same softmax, and each computes O^T for its own 256 latent
// dimensions (the value channels it holds).  The 2 x chunks CTAs of a
// sequence form one cluster (up to 16) that merges the chunks as above.
// ---------------------------------------------------------------------------
constexpr int kPairRegions = 5;                       // regions of 64 channels, at most
constexpr int kPairKvBytes = kPairRegions * kRegion;  // 80 KB
constexpr int kPairQBytes = kPairRegions * kQRegion;  // 40 KB
constexpr int kSxBytes = kEntries * kQRows * 4;       // 32 KB: the partner's S^T partial
constexpr uint32_t kPairTmemCols = 256;               // S^T: 64 cols, O^T: 2 x 64 cols

// Shared-memory address of the same object in CTA `rank` of the cluster.
__device__ inline uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(tc::smem_u32(p)), "r"(rank));
  return raddr;
}

// Bulk copy of `bytes` from this CTA's shared memory into another CTA's; the
// bytes complete a transaction on that CTA's mbarrier (which expects them).
__device__ inline void bulk_to_peer(uint32_t raddr, const void* src, uint32_t bytes, uint32_t rbar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(raddr), "r"(tc::smem_u32(src)), "r"(bytes), "r"(rbar)
               : "memory");
}

__device__ inline bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = tc::globaltimer_ns();
  while (true) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(tc::smem_u32(bar)), "r"(parity)
        : "memory");
    if (done) return true;
    if (tc::globaltimer_ns() - t0 > 200ull * 1000 * 1000) return false;
  }
}

// Remote arrival (release at cluster scope) on an mbarrier of another CTA.
__device__ inline void mbar_arrive_remote(uint32_t rbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar) : "memory");
}

// Cache row of entry slot `slot` of sequence b: a main-KV row (>= 0), SWA
// row r as -2 - r, or -1 for an empty slot.  t is the slot's Top-K index
// (slots < K); a bad index is reported when `report` is set.
__device__ inline int64_t entry_row(const AttnArgs& a, int b, int slot, int32_t t, int64_t n_ctx, int swl,
                                    bool report) {
  const int K = a.d.topk, W = a.d.swa;
  if (slot < K) {
    if (t >= 0 && t < n_ctx) {
      const int64_t r = kv_row(a.page_table, a.d, b, t, a.ws);
      return r < 0 ? -1 : r;
    }
    if (report && (t >= n_ctx || t < -1)) raise_err(a.ws, CSA2_DEV_TOPK_IDX);
    return -1;
  }
  return (slot < K + W && slot - K < swl) ? -2 - int64_t(slot - K) : -1;
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_pair_kernel(AttnArgs a, const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap swamap, int swa_tma_split) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* kv_s = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);   // nreg x 16 KB
  uint8_t* q_s = kv_s + kPairKvBytes;               // nreg x 8 KB; later P^T hi / lo
  float* sx = reinterpret_cast<float*>(q_s + kPairQBytes);   // [entry][head chunk], written by the partner
  float* sx_out = sx + kEntries * kQRows;           // this CTA's partial, copied to the partner
  __shared__ uint64_t bar_ld, bar_s, bar_o, bar_x, bar_ml, bar_zero;
  __shared__ uint32_t tmem_slot;
  __shared__ int64_t row_s[kEntries];               // >= 0 main row, -2 - r SWA row r, -1 empty
  __shared__ __align__(16) float red_m[4][4][16];
  __shared__ __align__(16) float red_l[4][4][16];
  __shared__ float fac_s[kQRows];                   // 2^(m_chunk - M) / L per head
  __shared__ __align__(16) float ml_all[kMaxClusterSplits][2][kQRows];   // every chunk's (m, l), base-2 m
  __shared__ __align__(16) float ml_mine[2][kQRows];                      // this chunk's, copied to all
  __shared__ bool ml_ok, z_ok;

  cg::cluster_group cl = cg::this_cluster();
  const int rank = int(cl.block_rank()), csize = int(cl.num_blocks());
  const int chunk = rank >> 1, half = rank & 1, S = csize >> 1;
  const int b = blockIdx.y;
  const int H = a.d.heads, K = a.d.topk, W = a.d.swa;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int nreg = half ? 5 : 4, reg0 = 4 * half;   // this CTA's regions of 64 channels (of 9)
  const bool paged = a.page_table != nullptr;
  const bool swa_tma = chunk == swa_tma_split;      // this chunk's rows are the SWA window
  // the chunk that finishes first (the TMA-loaded SWA window, else chunk 0)
  // zeroes the output and tells the other chunks of its half when it has
  const bool zero_cta = chunk == (swa_tma_split >= 0 ? swa_tma_split : 0);
  // set-up that touches no global memory, then wait for the previous kernel
  if (wid == 0) tc::tmem_alloc(&tmem_slot, kPairTmemCols);
  if (tid == 0) {
    tc::mbar_init(&bar_ld, 1);
    tc::mbar_init(&bar_s, 1);
    tc::mbar_init(&bar_o, 1);
    tc::mbar_init(&bar_x, 1);                        // the partner's S^T partial (32 KB)
    tc::mbar_init(&bar_ml, 1);                       // every chunk's (m, l) (S x 512 bytes)
    tc::mbar_init(&bar_zero, 1);                     // the zeroing chunk of this half is done
    tc::fence_mbar_init();
    // this CTA's own arrivals; the copies of the other CTAs bring the bytes
    tc::mbar_expect_tx(&bar_x, uint32_t(kSxBytes));
    tc::mbar_expect_tx(&bar_ml, uint32_t(S) * uint32_t(sizeof(ml_mine)));
  }
  // every CTA of the cluster must have started before another writes into
  // its shared memory: arrive now, wait before the first such write
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  pdl_wait();
  pdl_launch_dependents();
  // ---- loads that depend on nothing earlier in this kernel go out first:
  //      this half's query channels (and the window's rows) by TMA, the
  //      chunk's Top-K indices and the lengths ---------------------------------------
  if (tid == 0) {
    tc::mbar_expect_tx(&bar_ld, uint32_t(nreg) * (uint32_t(kQRegion) + (swa_tma ? uint32_t(kRegion) : 0u)));
    for (int kb = 0; kb < nreg; ++kb)
      tc::tma_load_2d(&qmap, q_s + kb * kQRegion, 64 * (reg0 + kb), b * H, &bar_ld);
    if (swa_tma)
      for (int kb = 0; kb < nreg; ++kb)
        tc::tma_load_2d(&swamap, kv_s + kb * kRegion, 64 * (reg0 + kb), b * W, &bar_ld);
  }
  auto topk_at = [&](int e) -> int32_t {
    const int slot = chunk * kEntries + e;
    return slot < K ? __ldg(a.topk + int64_t(b) * K + slot) : -1;
  };
  const int eg = tid >> 3;                          // this thread's gather entries: eg, eg + 64
  int32_t tg0 = -1, tg1 = -1;
  if (!swa_tma) {
    tg0 = topk_at(eg);
    tg1 = topk_at(eg + 64);
  }
  const int32_t trow = tid < kEntries ? topk_at(tid) : -1;
  int swl = __ldg(a.swa_len + b);
  const int64_t n_ctx = checked_ctx(a.ctx_len, a.d, b, paged, a.ws);
  if (swl < 0 || swl > W) {
    if (tid == 0 && half == 0) raise_err(a.ws, CSA2_DEV_SWA_LEN);
    swl = swl < 0 ? 0 : W;
  }
  if (tid < kEntries) row_s[tid] = entry_row(a, b, chunk * kEntries + tid, trow, n_ctx, swl, true);
  // ---- FP4 entries: gather (all loads first), dequantize to bf16 -------------------
  if (!swa_tma) {
    // latent: task = (entry, pair of 16-channel groups of this half); rope
    // (half 1): task = (entry, 16-byte chunk); entries eg and eg + 64
    const int64_t rr[2] = {entry_row(a, b, chunk * kEntries + eg, tg0, n_ctx, swl, false),
                           entry_row(a, b, chunk * kEntries + eg + 64, tg1, n_ctx, swl, false)};
    const int gp = 8 * half + (tid & 7), rc = tid & 7;
    uint4 cd[2], rp[2];
    uint32_t sc[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      cd[k] = make_uint4(0, 0, 0, 0);
      rp[k] = make_uint4(0, 0, 0, 0);
      sc[k] = 0;
      if (rr[k] >= 0) {
        cd[k] = __ldg(reinterpret_cast<const uint4*>(a.codes + rr[k] * kCodesPerRow) + gp);
        sc[k] = __ldg(reinterpret_cast<const uint16_t*>(a.scales + rr[k] * kScalesPerRow) + gp);
        if (half) rp[k] = __ldg(reinterpret_cast<const uint4*>(a.rope + rr[k] * kRope) + rc);
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int e = eg + 64 * k;
      if (rr[k] <= -2) continue;                     // SWA row: copied below
      uint32_t cw[4] = {cd[k].x, cd[k].y, cd[k].z, cd[k].w};
#pragma unroll
      for (int g = 0; g < 2; ++g) {                  // two 16-channel groups
        float s = e4m3_to_f32((sc[k] >> (8 * g)) & 0xFF);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t h2 = e2m1x2_to_f16x2_a((cw[2 * g + (i >> 2)] >> (8 * (i & 3))) & 0xFF);
          float lo = __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFF))) * s;
          float hi = __half2float(__ushort_as_half(uint16_t(h2 >> 16))) * s;
          w[i] = pack_bf16x2(lo, hi);
        }
        const int part = 2 * gp + g;                 // 16-channel group index 0..31
        const uint32_t region = (part >> 2) - reg0, ch0 = (part & 3) * 2;
        st_shared_v4(kv_s, region * kRegion + tc::sw128_offset(e, ch0), make_uint4(w[0], w[1], w[2], w[3]));
        st_shared_v4(kv_s, region * kRegion + tc::sw128_offset(e, ch0 + 1), make_uint4(w[4], w[5], w[6], w[7]));
      }
      if (half) st_shared_v4(kv_s, 4 * kRegion + tc::sw128_offset(e, rc), rp[k]);
    }
  }
  tc::tc_fence_before_sync();
  __syncthreads();
  tc::tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;
  if (!swa_tma) {
    // SWA rows of a chunk the window does not start on a 128-row boundary for
    const int nch = nreg * 8, c0 = reg0 * 8;          // this half's 16-byte chunks of a row
#pragma unroll 4
    for (int task = tid; task < kEntries * nch; task += kAttnThreads) {
      const int e = task / nch, c = task % nch;
      const int64_t r = row_s[e];
      if (r > -2) continue;
      uint4 v = __ldg(reinterpret_cast<const uint4*>(a.swa + (int64_t(b) * W + (-2 - r)) * kDqk) + c0 + c);
      st_shared_v4(kv_s, (c >> 3) * kRegion + tc::sw128_offset(e, c & 7), v);
    }
  }
  if (zero_cta) {
    for (int i = tid; i < H * 64; i += kAttnThreads) {
      const int h = i >> 6, q = i & 63;
      reinterpret_cast<float4*>(a.out + (int64_t(b) * H + h) * kLatent + half * 256)[q] =
          make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // every CTA has started
    // the zeros happen before every later reduce-add of this half
    if (tid < csize && (tid & 1) == half && (tid >> 1) != chunk)
      mbar_arrive_remote(cluster_addr(&bar_zero, uint32_t(tid)));
  }
  bool ok = tc::mbar_wait_bounded(&bar_ld, 0);
  if (swa_tma) {
    // window rows past swa_len (or past W) are not entries: zero them so that
    // P = 0 never meets a non-finite value
    const int nch = nreg * 8;
    for (int task = tid; task < kEntries * nch; task += kAttnThreads) {
      const int e = task / nch, c = task % nch;
      if (row_s[e] == -1) st_shared_v4(kv_s, (c >> 3) * kRegion + tc::sw128_offset(e, c & 7), make_uint4(0, 0, 0, 0));
    }
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before_sync();
  __syncthreads();

  // ---- S^T partial = KV_half . Q_half^T ------------------------------------------
  const uint32_t kv_addr = tc::smem_u32(kv_s), q_addr = tc::smem_u32(q_s);
  if (tid == 0) {
    tc::tc_fence_after_sync();
    constexpr uint32_t idS = tc::idesc_bf16(kEntries, kQRows, 0, 0);
    // descriptors are formed once; an offset of x bytes adds x/16 to the
    // start-address field (the operands lie below 256 KB, so it never carries)
    const uint64_t ad0 = tc::smem_desc(kv_addr, 16, 1024, 2), bd0 = tc::smem_desc(q_addr, 16, 1024, 2);
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
      const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
      tc::mma_bf16(tmem, ad0 + ((kb * kRegion + off) >> 4), bd0 + ((kb * kQRegion + off) >> 4), idS, ks > 0);
    }
    if (half) {
#pragma unroll
      for (int ks = 16; ks < 20; ++ks) {
        const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
        tc::mma_bf16(tmem, ad0 + ((kb * kRegion + off) >> 4), bd0 + ((kb * kQRegion + off) >> 4), idS, true);
      }
    }
    tc::mma_commit(&bar_s);
  }
  ok = tc::mbar_wait_bounded(&bar_s, 0) && ok;
  tc::tc_fence_after_sync();

  // ---- exchange the S^T partials within the pair ----------------------------------
  const int quarter = wid & 3, hg = wid >> 2;       // lanes 32*quarter.., heads 16*hg..
  const int e = quarter * 32 + lane;
  const bool valid = row_s[e] != -1;
  float x[16];
  tc::tmem_ld16(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(hg * 16), x);
  if (!zero_cta) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // every CTA has started
  // Each warp's part (its 32 rows x 16 heads) is one contiguous 2 KB block
  // of sx_out (block wid; the 16-byte slot i of lane l at 4l + (i ^ s_l),
  // s_l = (l >> 1) & 3, so that 8 consecutive lanes cover all banks), sent by
  // the warp itself as one bulk copy into the same block of the partner's sx
  // (the partner's warp wid holds the same rows and heads).
  const int sw = (lane >> 1) & 3;
  {
    float4* blk = reinterpret_cast<float4*>(sx_out) + wid * 128;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      blk[lane * 4 + (i ^ sw)] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      const float4* peer_blk = reinterpret_cast<const float4*>(sx) + wid * 128;   // the partner's sx, same block
      bulk_to_peer(cluster_addr(peer_blk, uint32_t(rank ^ 1)), blk, 2048u, cluster_addr(&bar_x, uint32_t(rank ^ 1)));
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
  }
  // every thread waits for the partner's 16 blocks itself
  ok = mbar_wait_cluster(&bar_x, 0) && ok;
  {
    const float4* src = reinterpret_cast<const float4*>(sx) + wid * 128;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = src[lane * 4 + (i ^ sw)];
      // own + partner: the same sum in both CTAs (fp32 addition commutes)
      x[4 * i] += v.x; x[4 * i + 1] += v.y; x[4 * i + 2] += v.z; x[4 * i + 3] += v.w;
    }
  }

  // ---- softmax over the 128 entries (TMEM lanes), identical in both halves ---------
  const float c2 = a.scale * 1.4426950408889634f;   // logits in base 2
#pragma unroll
  for (int j = 0; j < 16; ++j) x[j] = valid ? x[j] * c2 : -INFINITY;
  {
    const float m = butterfly16<true>(x, lane);
    if ((lane & 1) == 0) red_m[hg][quarter][butterfly_index(lane)] = m;
  }
  __syncthreads();
  float p[16];
#pragma unroll
  for (int j4 = 0; j4 < 4; ++j4) {
    float4 m4[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) m4[q] = reinterpret_cast<const float4*>(&red_m[hg][q][0])[j4];
    const float Mj[4] = {fmaxf(fmaxf(m4[0].x, m4[1].x), fmaxf(m4[2].x, m4[3].x)),
                         fmaxf(fmaxf(m4[0].y, m4[1].y), fmaxf(m4[2].y, m4[3].y)),
                         fmaxf(fmaxf(m4[0].z, m4[1].z), fmaxf(m4[2].z, m4[3].z)),
                         fmaxf(fmaxf(m4[0].w, m4[1].w), fmaxf(m4[2].w, m4[3].w))};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = 4 * j4 + i;
      p[j] = (Mj[i] == -INFINITY || x[j] == -INFINITY) ? 0.0f : exp2f(x[j] - Mj[i]);
    }
  }
  {
    const float l = butterfly16<false>(p, lane);
    if ((lane & 1) == 0) red_l[hg][quarter][butterfly_index(lane)] = l;
  }
  // P^T rows (entry e) as bf16 hi and lo parts; the query buffer is free (the
  // S^T MMAs completed before this)
  uint8_t* p_hi = q_s;
  uint8_t* p_lo = q_s + kRegion;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    uint32_t wh[4], wl[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float v0 = p[8 * t + 2 * i], v1 = p[8 * t + 2 * i + 1];
      uint32_t hb = pack_bf16x2(v0, v1);
      float h0 = __uint_as_float(hb << 16), h1 = __uint_as_float(hb & 0xFFFF0000u);
      wh[i] = hb;
      wl[i] = pack_bf16x2(v0 - h0, v1 - h1);
    }
    uint32_t off = tc::sw128_offset(e, hg * 2 + t);
    st_shared_v4(p_hi, off, make_uint4(wh[0], wh[1], wh[2], wh[3]));
    st_shared_v4(p_lo, off, make_uint4(wl[0], wl[1], wl[2], wl[3]));
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before_sync();
  __syncthreads();

  // ---- O^T = V_half^T . P^T  (this half's 2 M-tiles of 128 dims; hi and lo) --------
  if (tid == 0) {
    tc::tc_fence_after_sync();
    constexpr uint32_t idO = tc::idesc_bf16(kEntries, kQRows, 1, 1);
    const uint64_t av0 = tc::smem_desc(kv_addr, kRegion, 1024, 2);
    const uint64_t bp0[2] = {tc::smem_desc(tc::smem_u32(p_hi), kRegion, 1024, 2),
                             tc::smem_desc(tc::smem_u32(p_lo), kRegion, 1024, 2)};
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
      for (int part = 0; part < 2; ++part) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc::mma_bf16(tmem + 64 + 64 * mt, av0 + (((2 * mt) * kRegion + ks * 2048) >> 4),
                       bp0[part] + ((ks * 2048) >> 4), idO, part > 0 || ks > 0);
      }
    }
    tc::mma_commit(&bar_o);
  }
  // this chunk's (m, l) per head: half 0 copies it into every CTA of the cluster
  if (half == 0 && quarter == 0) {
    if (lane < 16) {
      const int h = hg * 16 + lane;
      ml_mine[0][h] = fmaxf(fmaxf(red_m[hg][0][lane], red_m[hg][1][lane]), fmaxf(red_m[hg][2][lane], red_m[hg][3][lane]));
      ml_mine[1][h] = red_l[hg][0][lane] + red_l[hg][1][lane] + red_l[hg][2][lane] + red_l[hg][3][lane];
    }
    tc::fence_proxy_async_smem();
    asm volatile("bar.sync 2, 128;" ::: "memory");   // the 4 warps of quarter 0
    if (wid == 0 && lane < csize) {
      bulk_to_peer(cluster_addr(&ml_all[chunk][0][0], uint32_t(lane)), &ml_mine[0][0], uint32_t(sizeof(ml_mine)),
                   cluster_addr(&bar_ml, uint32_t(lane)));
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
  }

  // ---- merge over the cluster -------------------------------------------------------
  if (tid == 32) ml_ok = mbar_wait_cluster(&bar_ml, 0);     // every chunk's (m, l)
  if (tid == 64) z_ok = zero_cta || mbar_wait_cluster(&bar_zero, 0);
  __syncthreads();
  ok = ml_ok && z_ok && ok;
  if (tid < kQRows) {
    float mr[kMaxClusterSplits], lr[kMaxClusterSplits];
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < kMaxClusterSplits; ++r) {
      mr[r] = (r < S && tid < H) ? ml_all[r][0][tid] : -INFINITY;
      lr[r] = (r < S && tid < H) ? ml_all[r][1][tid] : 0.0f;
      M = fmaxf(M, mr[r]);
    }
    float L = 0.0f;
#pragma unroll
    for (int r = 0; r < kMaxClusterSplits; ++r)
      if (mr[r] != -INFINITY) L += lr[r] * exp2f(mr[r] - M);
    float ms = -INFINITY;
#pragma unroll
    for (int r = 0; r < kMaxClusterSplits; ++r) ms = r == chunk ? mr[r] : ms;
    fac_s[tid] = (ms == -INFINITY || !(L > 0.0f)) ? 0.0f : exp2f(ms - M) / L;
    if (rank == 0 && tid < H)
      a.lse[int64_t(b) * H + tid] = L > 0.0f ? M * 0.6931471805599453f + logf(L) : -INFINITY;
  }
  ok = tc::mbar_wait_bounded(&bar_o, 0) && ok;
  tc::tc_fence_after_sync();
  __syncthreads();
  if (!ok && tid == 0) raise_err(a.ws, CSA2_DEV_TIMEOUT);
  // scaled O^T added into this half's output dimensions straight from tensor
  // memory: for one head the 32 lanes of a warp hold 32 consecutive dims
#pragma unroll 1
  for (int mt = 0; mt < 2; ++mt) {
    float o[16];
    tc::tmem_ld16(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(64 + 64 * mt + hg * 16), o);
    float* dst = a.out + int64_t(b) * H * kLatent + half * 256 + mt * 128 + quarter * 32 + lane;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int h = hg * 16 + j;
      if (h < H)
        asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst + int64_t(h) * kLatent), "f"(o[j] * fac_s[h])
                     : "memory");
    }
  }
  tc::tc_fence_before_sync();
  __syncthreads();
  if (wid == 0) tc::tmem_dealloc(tmem, kPairTmemCols);
  // the bulk copies this thread committed (a warp's sx_out block, warp 0's
  // ml_mine copies) have read their source before the CTA exits
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__global__ void __launch_bounds__(128) attn_combine_kernel(AttnArgs a) {
  const int h = blockIdx.x, b = blockIdx.y, H = a.d.heads, S = a.L.splits;
  pdl_wait();
  pdl_launch_dependents();
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

size_t attn_smem_bytes(int) { return size_t(kKvBytes) + size_t(kQBytes) + 1024; }

static PFN_cuTensorMapEncodeTiled_v12000 attn_encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [rows][576] bf16 rows of 1152 bytes, boxes of 64 channels x box_rows.
static bool encode_rows_map(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  return encode_2d_cached(attn_encode_fn(), map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, uint64_t(kDqk), rows,
                          uint64_t(kDqk) * 2, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

cudaError_t launch_attention(AttnArgs a, cudaStream_t st) {
  CUtensorMap qmap, swamap;
  if (!encode_rows_map(&qmap, a.q, uint64_t(a.batch) * a.d.heads, kQRows)) return cudaErrorInvalidValue;
  // the window is loaded by TMA when it starts a 128-entry split
  int swa_split = -1;
  if (a.d.swa > 0 && a.d.swa <= kEntries && a.d.topk % kEntries == 0) swa_split = a.d.topk / kEntries;
  swamap = qmap;
  if (swa_split >= 0 &&
      !encode_rows_map(&swamap, a.swa, uint64_t(a.batch) * a.d.swa, kEntries))
    return cudaErrorInvalidValue;
  size_t smem = attn_smem_bytes(a.d.heads);
  if (!attn_uses_partials(a.d)) {
    // one cluster of 2 x chunks CTAs per sequence; the merge happens inside it
    const size_t psmem = size_t(kPairKvBytes) + size_t(kPairQBytes) + 2 * size_t(kSxBytes) + 1024;
    static KernelAttrs done;
    cudaError_t e = prepare_kernel(attn_pair_kernel, psmem, true, done);
    if (e != cudaSuccess) return e;
    CSA2_PROFILED(st, "attn_pair_tc",
                  (e = launch_pdl(attn_pair_kernel, dim3(unsigned(2 * a.L.splits), unsigned(a.batch), 1),
                                  dim3(kAttnThreads), psmem, st, unsigned(2 * a.L.splits), a, qmap, swamap,
                                  swa_split)));
    return e;
  }
  static KernelAttrs done_partial;
  cudaError_t e = prepare_kernel(attn_partial_tc_kernel, smem, false, done_partial);
  if (e != cudaSuccess) return e;
  CSA2_PROFILED(st, "attn_partial_tc",
                (e = launch_pdl(attn_partial_tc_kernel, dim3(unsigned(a.L.splits), unsigned(a.batch)),
                                dim3(kAttnThreads), smem, st, 1, a, qmap, swamap, swa_split)));
  if (e != cudaSuccess) return e;
  CSA2_PROFILED(st, "attn_combine", (e = launch_pdl(attn_combine_kernel, dim3(unsigned(a.d.heads), unsigned(a.batch)),
                                                    dim3(128), 0, st, 1, a)));
  return e;
}

}  // namespace csa2
