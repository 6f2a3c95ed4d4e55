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
// attn_cluster_kernel (K + W <= 1024, the usual case): one CTA per (sequence,
// group of 32 heads, chunk of 128 entries) with all 576 channels of its
// entries; the chunks of a (sequence, head group) form one thread-block
// cluster: every chunk copies its per-head (m_s, l_s) into every CTA's shared
// memory, on an mbarrier that counts the bytes; chunk 0 zeroes the head
// group's output rows early and signals the other chunks; each CTA then forms
// M and L, scales its O^T part and adds it into the output with coalesced
// reduce-adds (red.global.add.f32) straight from tensor memory.  The order of
// the additions is not fixed, so the last bits of the output may differ
// between runs.  In Reuse mode the entries are gathered before the kernel
// waits for the one before it (see the kernel's comment).
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
// Cluster kernel (K + W <= 1024, the usual case).  One CTA per (sequence,
// group of 32 heads, chunk of 128 entry slots); the chunks of one (sequence,
// head group) form a thread-block cluster (up to 8 CTAs) that merges them.
// A CTA holds all 576 key channels of its 128 entries (144 KB of bf16) and
// the query of its 32 heads (36 KB), so no partial scores are exchanged:
//   * S^T[128 entries x 32 heads] = KV . Q^T (M = 128, N = 32, K = 576), the
//     K steps spread round-robin over 4 tensor-memory accumulators, each
//     issued by its own thread (the softmax adds the 4 partial sums);
//   * softmax over the 128 entries (TMEM lanes; 16 warps, 8 heads each);
//   * P^T stored K-major as bf16 hi and lo parts side by side: rows 0..31
//     hold the hi parts of the 32 heads, rows 32..63 the lo parts;
//   * O^T[512 dims x (hi | lo) 64] = V^T . [P_hi | P_lo]^T: 4 M-tiles, N = 64,
//     K = 128 (one instruction covers both parts), each tile's MMAs issued
//     by its own thread;
//   * merge: every chunk copies its (m, l) into every CTA of the cluster
//     (warp 1, while the O MMAs are issued); every chunk zeroes its share
//     of the head group's output rows and signals the others; each CTA adds
//     its scaled O (hi + lo) into the output with coalesced reduce-adds
//     (red.global.add.f32) straight from tensor memory.
// Chunk c holds the Top-K slots [K c / S, K (c + 1) / S) and then window
// rows up to 128 entries (the window filled into the chunks in order), so
// that every CTA loads a share of the window.  One CTA per SM (its shared
// memory), as every tensor-memory kernel of the library.  In Reuse mode (the
// indices and the main-KV cache come from earlier work on the stream) the
// Top-K indices are read and the entries gathered and dequantized before
// griddepcontrol.wait; the query, the window and the outputs are read or
// written only after it (an L2 prefetch of the query and window rows is
// issued before it), with coalesced 16-byte loads by all threads.
// ---------------------------------------------------------------------------
constexpr int kCEntries = kEntries;                  // entry slots per CTA (= MMA M)
constexpr int kCHeads = 32;                          // heads per CTA (MMA N)
constexpr int kCQRegion = kCHeads * 128;             // 64 channels x 32 heads: 4 KB
constexpr int kCQBytes = 9 * kCQRegion;              // 36 KB (later P^T hi / lo)
constexpr int kCPRegion = 2 * kCHeads * 128;         // P^T hi | lo: 64 rows x 64 entries: 8 KB
constexpr int kSAcc = 4;                            // S^T partial accumulators
constexpr uint32_t kCTmemCols = 512;                 // S^T: 4 x 32 cols, O^T: 4 x 64 cols (hi | lo)
constexpr uint32_t kCOCol = kSAcc * kCHeads;         // first O^T column
static_assert(2 * kCPRegion <= kCQBytes, "P^T (two regions of 64 entries) fits the query buffer");
static_assert(kCOCol + 4 * 2 * kCHeads <= kCTmemCols, "tensor-memory columns");

struct ClusterSmall {
  uint64_t bar_s, bar_o, bar_ml, bar_zero;
  uint32_t valid[kCEntries / 32];                    // bit e: entry slot e holds an entry
  uint32_t tmem_slot;
  int32_t ok_ml, ok_z;
  __align__(16) float red_m[4][4][8];                // [head octet][lane quarter][head]
  float red_l[4][4][8];
  float fac[kCHeads];                                // 2^(m_chunk - M) / L per head
  __align__(16) float ml_mine[2][kCHeads];           // this chunk's (m, l), base-2 m
  __align__(16) float ml_all[kMaxClusterSplits][2][kCHeads];   // every chunk's (m, l)
  int64_t rows[kCEntries];                           // cache row of each entry slot (cluster_gather)
};

size_t cluster_smem_bytes() { return 1024 + size_t(kKvBytes) + size_t(kCQBytes) + sizeof(ClusterSmall); }

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

// Reduces 8 values per lane over the warp (reduce-scatter): returns the
// reduction of value index octet_index(lane), held by lanes 4i .. 4i+3.
__device__ inline int octet_index(int lane) {
  return (((lane >> 4) & 1) << 2) | (((lane >> 3) & 1) << 1) | ((lane >> 2) & 1);
}

template <bool kMax>
__device__ inline float butterfly8(const float (&v)[8], int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float y[4], z[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b4 ? v[4 + i] : v[i], give = b4 ? v[i] : v[4 + i];
    y[i] = op(keep, __shfl_xor_sync(0xFFFFFFFFu, give, 16));
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b3 ? y[2 + i] : y[i], give = b3 ? y[i] : y[2 + i];
    z[i] = op(keep, __shfl_xor_sync(0xFFFFFFFFu, give, 8));
  }
  const float keep = b2 ? z[1] : z[0], give = b2 ? z[0] : z[1];
  float u = op(keep, __shfl_xor_sync(0xFFFFFFFFu, give, 4));
  u = op(u, __shfl_xor_sync(0xFFFFFFFFu, u, 2));
  return op(u, __shfl_xor_sync(0xFFFFFFFFu, u, 1));
}

// Coalesced gather: a half-warp reads one entry (its 256 code bytes, 32 scale
// bytes and 128 rope bytes), so that a warp instruction touches the lines of
// two entries rather than of 32.  Lane p (0..15) of the half-warp owns the
// 16-byte chunk c = p % 8 (8 channels) of the latent regions p / 8 + 2 j
// (j = 0..3): each of its four stores is then one of 8 chunk positions of
// the swizzled rows across the half-warp (no bank conflicts), and each load
// instruction reads 64 contiguous code bytes of the entry.  Thread piece k
// (0..3) is entry 2 (warp + 16 k) + lane / 16.
struct GatherCo {
  uint32_t cw[4][4];                                 // [entry piece][region j]: 8 FP4 codes
  uint32_t sb[4];                                    // [entry piece]: byte j = the scale of region j's chunk
  uint4 rp[4];                                       // rope chunk p (lanes p < 8)
  uint32_t skip;                                     // bit k: piece k is a window row (written with the window)
};

__device__ inline void gather_load_co(const AttnArgs& a, GatherCo& g, const int64_t* rows, int nm, int nw,
                                      int wid, int lane) {
  const int p = lane & 15, c = p & 7, r0 = p >> 3;
  g.skip = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = 2 * (wid + 16 * k) + (lane >> 4);
    const int64_t row = e < nm ? rows[e] : -1;
    if (e >= nm && e < nm + nw) g.skip |= 1u << k;
    g.sb[k] = 0;
    g.rp[k] = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < 4; ++j) g.cw[k][j] = 0;
    if (row >= 0) {
      const uint8_t* cp = a.codes + row * kCodesPerRow;
      const uint8_t* sp = a.scales + row * kScalesPerRow;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = r0 + 2 * j;                    // region: latent channels 64 r .. 64 r + 63
        g.cw[k][j] = __ldg(reinterpret_cast<const uint32_t*>(cp + 32 * r + 4 * c));
        g.sb[k] |= uint32_t(__ldg(sp + 4 * r + (c >> 1))) << (8 * j);
      }
      if (p < 8) g.rp[k] = __ldg(reinterpret_cast<const uint4*>(a.rope + row * kRope) + p);
    }
  }
}

__device__ inline void gather_store_co(uint8_t* kv_s, const GatherCo& g, int wid, int lane) {
  const int p = lane & 15, c = p & 7, r0 = p >> 3;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if ((g.skip >> k) & 1) continue;
    const int e = 2 * (wid + 16 * k) + (lane >> 4);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float sc = e4m3_to_f32((g.sb[k] >> (8 * j)) & 0xFF);
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t h2 = e2m1x2_to_f16x2_a((g.cw[k][j] >> (8 * i)) & 0xFF);
        w[i] = pack_bf16x2(__half2float(__ushort_as_half(uint16_t(h2 & 0xFFFF))) * sc,
                           __half2float(__ushort_as_half(uint16_t(h2 >> 16))) * sc);
      }
      st_shared_v4(kv_s + (r0 + 2 * j) * kRegion, tc::sw128_offset(e, c), make_uint4(w[0], w[1], w[2], w[3]));
    }
    if (p < 8) st_shared_v4(kv_s + 8 * kRegion, tc::sw128_offset(e, p), g.rp[k]);
  }
}

// The chunk's FP4 main-KV entries, dequantized exactly to bf16 into the
// 128-byte swizzled KV tile: threads 0..127 resolve entry tid's cache row into
// rows_s (Top-K slot m0 + e for e < nm; -2 - r for window row r = w0 + e - nm,
// written later; -1: no entry, its tile row zeroed), then every thread loads
// and writes its four coalesced pieces.  Returns the row of entry tid % 128.
__device__ inline int64_t cluster_gather(const AttnArgs& a, uint8_t* kv_s, int64_t* rows_s, int b, int m0, int nm,
                                         int w0, int nw, int64_t n_ctx, int tid) {
  const int K = a.d.topk;
  if (tid < kCEntries) {
    const int e = tid;
    int64_t row = -1;
    if (e < nm) {
      const int32_t t = __ldg(a.topk + int64_t(b) * K + m0 + e);
      if (t >= 0 && t < n_ctx) {
        row = kv_row(a.page_table, a.d, b, t, a.ws);
        if (row < 0) row = -1;
      } else if (t >= n_ctx || t < -1) {
        raise_err(a.ws, CSA2_DEV_TOPK_IDX);
      }
    } else if (e < nm + nw) {
      row = -2 - int64_t(w0 + e - nm);
    }
    rows_s[e] = row;
  }
  __syncthreads();
  GatherCo g;
  gather_load_co(a, g, rows_s, nm, nw, tid >> 5, tid & 31);
  gather_store_co(kv_s, g, tid >> 5, tid & 31);
  return rows_s[tid & (kCEntries - 1)];
}

__global__ void __launch_bounds__(kAttnThreads, 1) attn_cluster_kernel(AttnArgs a, int early) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* kv_s = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);   // 9 x 16 KB
  uint8_t* q_s = kv_s + kKvBytes;                    // 9 x 4 KB; later P^T hi / lo
  ClusterSmall& sm = *reinterpret_cast<ClusterSmall*>(q_s + kCQBytes);

  cg::cluster_group cl = cg::this_cluster();
  const int chunk = int(cl.block_rank()), S = int(cl.num_blocks());
  const int nhg = (a.d.heads + kCHeads - 1) / kCHeads;
  // blockIdx.y: (sequence, query of the sequence, head group); query qi of a
  // multi-query call sees the window rows below swa_len - (q_len - 1 - qi)
  const int qrow = blockIdx.y / nhg, hg = blockIdx.y % nhg;
  const int b = qrow / a.q_len, qi = qrow % a.q_len;
  const int H = a.d.heads, K = a.d.topk, W = a.d.swa;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool paged = a.page_table != nullptr;
  const bool lse_cta = chunk == 0;                   // writes the head group's lse
  const int h0 = hg * kCHeads, nh = min(kCHeads, H - h0);
  const int m0 = attn_chunk_main_lo(K, chunk, S), nm = attn_chunk_main_lo(K, chunk + 1, S) - m0;
  int w0, nw;
  attn_chunk_window(K, W, chunk, S, w0, nw);
  // ---- set-up that touches no global memory -----------------------------------------
  if (wid == 0) tc::tmem_alloc(&sm.tmem_slot, kCTmemCols);
  if (tid == 0) {
    tc::mbar_init(&sm.bar_s, kSAcc);                 // one commit per MMA-issuing thread
    tc::mbar_init(&sm.bar_o, 4);
    tc::mbar_init(&sm.bar_ml, 1);                    // every chunk's (m, l): S x 256 bytes
    tc::mbar_init(&sm.bar_zero, S > 1 ? S - 1 : 1);  // the other chunks have zeroed their rows
    tc::fence_mbar_init();
    tc::mbar_expect_tx(&sm.bar_ml, uint32_t(S) * uint32_t(sizeof(sm.ml_mine)));
  }
  __syncwarp();
  // every CTA of the cluster must have started before another writes into
  // its shared memory: arrive now, wait before the first such write
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  // ---- the chunk's main-KV entries: before the wait in Reuse mode -----------------
  int64_t row = -1;
  {
    // L2 prefetch (a hint: nothing is read into the SM) of what is read right
    // after the wait: the window length, this head group's query rows (36 KB)
    // and this chunk's window rows; the reads themselves follow the wait
    const char* qb = reinterpret_cast<const char*>(a.q + (int64_t(qrow) * H + h0) * kDqk);
    const char* wb = reinterpret_cast<const char*>(a.swa + (int64_t(b) * W + w0) * kDqk);
    const int qlines = (nh * kDqk * 2 + 127) / 128, wlines = (nw * kDqk * 2 + 127) / 128;
    for (int i = tid; i < qlines + wlines; i += kAttnThreads) {
      const char* pf = i < qlines ? qb + 128 * i : wb + 128 * (i - qlines);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(pf));
    }
    if (tid == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.swa_len + b));
  }
  if (early) row = cluster_gather(a, kv_s, sm.rows, b, m0, nm, w0, nw, checked_ctx(a.ctx_len, a.d, b, paged, a.ws), tid);
  pdl_wait();
  pdl_launch_dependents();
  // ---- after the wait: the window length, this head group's query (32 rows
  //      x 576 channels, one contiguous 36 KB run) and this chunk's window rows
  //      (nw contiguous rows), every load issued before any is used ---------------
  int swl = __ldg(a.swa_len + b);
  constexpr int kQVec = kCHeads * (kDqk / 8);        // 16-byte pieces of the query rows
  constexpr int kQPer = (kQVec + kAttnThreads - 1) / kAttnThreads;
  const uint4* qsrc = reinterpret_cast<const uint4*>(a.q + (int64_t(qrow) * H + h0) * kDqk);
  uint4 qv[kQPer];
#pragma unroll
  for (int k = 0; k < kQPer; ++k) {
    const int i = tid + k * kAttnThreads;
    qv[k] = (i < kQVec && i / (kDqk / 8) < nh) ? __ldg(qsrc + i) : make_uint4(0, 0, 0, 0);
  }
  constexpr int kWPer = 8;                           // window pieces per thread per batch
  const int nwv = nw * (kDqk / 8);
  const uint4* wsrc = reinterpret_cast<const uint4*>(a.swa + (int64_t(b) * W + w0) * kDqk);
  uint4 wv[kWPer];
#pragma unroll
  for (int k = 0; k < kWPer; ++k) {
    const int i = tid + k * kAttnThreads;
    wv[k] = i < nwv ? __ldg(wsrc + i) : make_uint4(0, 0, 0, 0);
  }
  if (!early) row = cluster_gather(a, kv_s, sm.rows, b, m0, nm, w0, nw, checked_ctx(a.ctx_len, a.d, b, paged, a.ws), tid);
  {
    // this chunk's share of the head group's output rows: zeros
    const int z0 = nh * chunk / S, z1 = nh * (chunk + 1) / S;
    float4* orow = reinterpret_cast<float4*>(a.out + (int64_t(qrow) * H + h0 + z0) * kLatent);
    for (int i = tid; i < (z1 - z0) * 128; i += kAttnThreads) orow[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (swl < 0 || swl > W) {
    if (tid == 0 && chunk == 0 && hg == 0 && qi == 0) raise_err(a.ws, CSA2_DEV_SWA_LEN);
    swl = swl < 0 ? 0 : W;
  }
  swl = max(0, swl - (a.q_len - 1 - qi));            // the later queries' rows are not visible
  // query pieces into the swizzled K-major tile [region][head row]
#pragma unroll
  for (int k = 0; k < kQPer; ++k) {
    const int i = tid + k * kAttnThreads;
    if (i < kQVec) {
      const int h = i / (kDqk / 8), j = i % (kDqk / 8);
      st_shared_v4(q_s, (j >> 3) * kCQRegion + tc::sw128_offset(h, j & 7), qv[k]);
    }
  }
  // window rows as entries nm .. nm + nw - 1 (rows at or past swa_len:
  // zeros); more than one batch only when a chunk holds over 56 window rows
  for (int base = 0; base < nwv; base += kWPer * kAttnThreads) {
    if (base > 0) {
#pragma unroll
      for (int k = 0; k < kWPer; ++k) {
        const int i = base + tid + k * kAttnThreads;
        wv[k] = i < nwv ? __ldg(wsrc + i) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int k = 0; k < kWPer; ++k) {
      const int i = base + tid + k * kAttnThreads;
      if (i < nwv) {
        const int r = i / (kDqk / 8), j = i % (kDqk / 8);
        st_shared_v4(kv_s, (j >> 3) * kRegion + tc::sw128_offset(nm + r, j & 7),
                     w0 + r < swl ? wv[k] : make_uint4(0, 0, 0, 0));
      }
    }
  }
  // entry slot e holds an entry: a main row, or a window row below swa_len
  const bool has = row >= 0 || (row <= -2 && -2 - row < swl);
  {
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, has);
    if (tid < kCEntries && lane == 0) sm.valid[tid >> 5] = m;
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before_sync();
  __syncthreads();
  tc::tc_fence_after_sync();
  const uint32_t tmem = sm.tmem_slot;

  // ---- S^T = KV . Q^T: lane 0 of warps 0..3 each issues the 9 K steps of one
  //      of 4 accumulators (K step 4 kb + k4 into accumulator k4) ----------------------
  const uint32_t kv_addr = tc::smem_u32(kv_s), q_addr = tc::smem_u32(q_s);
  if (wid < kSAcc && lane == 0) {
    constexpr uint32_t idS = tc::idesc_bf16(kCEntries, kCHeads, 0, 0);
    const uint64_t ad0 = tc::smem_desc(kv_addr, 16, 1024, 2), bd0 = tc::smem_desc(q_addr, 16, 1024, 2);
    const int k4 = wid;
#pragma unroll
    for (int kb = 0; kb < 9; ++kb) {
      const uint32_t off = uint32_t(kb * kRegion + k4 * 32), qoff = uint32_t(kb * kCQRegion + k4 * 32);
      tc::mma_bf16(tmem + uint32_t(k4 * kCHeads), ad0 + (off >> 4), bd0 + (qoff >> 4), idS, kb > 0);
    }
    tc::mma_commit(&sm.bar_s);
  }
  __syncwarp();
  // the cluster has started (warps 1 and 2, which write into other CTAs);
  // this chunk's zeros precede the others' reduce-adds (warp 2 signals)
  if (wid == 1 || wid == 2) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  if (wid == 2 && S > 1 && lane < S && lane != chunk) mbar_arrive_remote(cluster_addr(&sm.bar_zero, uint32_t(lane)));
  __syncwarp();
  bool ok = tc::mbar_wait_bounded(&sm.bar_s, 0);
  tc::tc_fence_after_sync();

  // ---- softmax over the 128 entries (TMEM lanes): 16 warps, 8 heads each ---------------
  const int quarter = wid & 3, oct = wid >> 2;       // lanes 32 quarter.., heads 8 oct..
  const int e = quarter * 32 + lane;
  uint8_t* p_s = q_s;                                // the query is no longer read (S^T done)
  {
    float x[8];
    {
      const uint32_t ta = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(oct * 8);
      float x1[8], x2[8], x3[8];
      tc::tmem_ld8(ta, x);
      tc::tmem_ld8(ta + kCHeads, x1);
      tc::tmem_ld8(ta + 2 * kCHeads, x2);
      tc::tmem_ld8(ta + 3 * kCHeads, x3);
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = (x[j] + x1[j]) + (x2[j] + x3[j]);
    }
    const bool v_e = (sm.valid[e >> 5] >> (e & 31)) & 1;
    const float c2 = a.scale * 1.4426950408889634f;   // logits in base 2
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = v_e ? x[j] * c2 : -INFINITY;
    {
      float mx[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(mx[j]) : "f"(x[j]));
      if (lane == 0) {
        float4* dst = reinterpret_cast<float4*>(&sm.red_m[oct][quarter][0]);
        dst[0] = make_float4(mx[0], mx[1], mx[2], mx[3]);
        dst[1] = make_float4(mx[4], mx[5], mx[6], mx[7]);
      }
    }
    __syncthreads();
    float p[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float Mj = fmaxf(fmaxf(sm.red_m[oct][0][j], sm.red_m[oct][1][j]),
                             fmaxf(sm.red_m[oct][2][j], sm.red_m[oct][3][j]));
      p[j] = (Mj == -INFINITY || x[j] == -INFINITY) ? 0.0f : exp2f(x[j] - Mj);
    }
    const float l = butterfly8<false>(p, lane);
    if ((lane & 3) == 0) sm.red_l[oct][quarter][octet_index(lane)] = l;
    // P^T[row][entry], K-major in two regions of 64 entries: row h the hi
    // bf16 part of head h, row 32 + h its lo part (2-byte stores: the 32
    // lanes write 64 consecutive bytes of a row)
    uint8_t* reg = p_s + (e >> 6) * kCPRegion;
    const uint32_t ch = uint32_t((e >> 3) & 7), el = uint32_t(e & 7) * 2;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int h = oct * 8 + j;
      const uint32_t hb = pack_bf16x2(p[j], 0.0f);
      const float hv = __uint_as_float(hb << 16);
      *reinterpret_cast<uint16_t*>(reg + tc::sw128_offset(uint32_t(h), ch) + el) = uint16_t(hb & 0xFFFF);
      *reinterpret_cast<uint16_t*>(reg + tc::sw128_offset(uint32_t(kCHeads + h), ch) + el) =
          uint16_t(pack_bf16x2(p[j] - hv, 0.0f) & 0xFFFF);
    }
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before_sync();
  __syncthreads();
  tc::tc_fence_after_sync();

  // ---- O^T = V^T . [P_hi | P_lo]^T  (4 M-tiles of 128 dims, N = 64, K = 128):
  //      lane 0 of warps 0, 2, 3, 4 each issues one tile's 8 K steps -------------------
  if ((wid == 0 || (wid >= 2 && wid <= 4)) && lane == 0) {
    constexpr uint32_t idO = tc::idesc_bf16(kCEntries, 2 * kCHeads, 1, 0);
    const uint64_t bp0 = tc::smem_desc(tc::smem_u32(p_s), 16, 1024, 2);
    const uint64_t av0 = tc::smem_desc(kv_addr, kRegion, 1024, 2);
    const int mt = wid == 0 ? 0 : wid - 1;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_bf16(tmem + kCOCol + 64 * mt, av0 + (((2 * mt) * kRegion + ks * 2048) >> 4),
                   bp0 + (((ks >> 2) * kCPRegion + (ks & 3) * 32) >> 4), idO, ks > 0);
    tc::mma_commit(&sm.bar_o);
  }
  __syncwarp();
  // this chunk's (m, l) per head, copied into every CTA of the cluster by
  // warp 1 while the O MMAs are issued
  if (wid == 1) {
    const int o8 = lane >> 3, j = lane & 7;
    sm.ml_mine[0][lane] = fmaxf(fmaxf(sm.red_m[o8][0][j], sm.red_m[o8][1][j]),
                                fmaxf(sm.red_m[o8][2][j], sm.red_m[o8][3][j]));
    sm.ml_mine[1][lane] = (sm.red_l[o8][0][j] + sm.red_l[o8][1][j]) + (sm.red_l[o8][2][j] + sm.red_l[o8][3][j]);
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane < S) {
      bulk_to_peer(cluster_addr(&sm.ml_all[chunk][0][0], uint32_t(lane)), &sm.ml_mine[0][0],
                   uint32_t(sizeof(sm.ml_mine)), cluster_addr(&sm.bar_ml, uint32_t(lane)));
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
    __syncwarp();
  }

  // ---- merge over the cluster ------------------------------------------------------------
  if (tid == 32) sm.ok_ml = mbar_wait_cluster(&sm.bar_ml, 0);
  if (tid == 64) sm.ok_z = S == 1 || mbar_wait_cluster(&sm.bar_zero, 0);
  __syncthreads();
  ok = sm.ok_ml && sm.ok_z && ok;
  if (tid < kCHeads) {
    float M = -INFINITY;
    for (int r = 0; r < S; ++r) M = fmaxf(M, sm.ml_all[r][0][tid]);
    float L = 0.0f;
    for (int r = 0; r < S; ++r) {
      const float mr = sm.ml_all[r][0][tid];
      if (mr != -INFINITY) L += sm.ml_all[r][1][tid] * exp2f(mr - M);
    }
    const float ms = sm.ml_all[chunk][0][tid];
    sm.fac[tid] = (ms == -INFINITY || !(L > 0.0f)) ? 0.0f : exp2f(ms - M) / L;
    if (lse_cta && tid < nh)
      a.lse[int64_t(qrow) * H + h0 + tid] = L > 0.0f ? M * 0.6931471805599453f + logf(L) : -INFINITY;
  }
  ok = tc::mbar_wait_bounded(&sm.bar_o, 0) && ok;
  tc::tc_fence_after_sync();
  __syncthreads();
  if (!ok && tid == 0) raise_err(a.ws, CSA2_DEV_TIMEOUT);
  // scaled O (hi + lo parts) added into the output straight from tensor
  // memory: for one head a warp's 32 lanes hold 32 consecutive dims
  float* dst0 = a.out + (int64_t(qrow) * H + h0) * kLatent + quarter * 32 + lane;
#pragma unroll 1
  for (int mt = 0; mt < 4; ++mt) {
    float hi[8], lo[8];
    const uint32_t ta = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(kCOCol + 64 * mt + oct * 8);
    tc::tmem_ld8(ta, hi);
    tc::tmem_ld8(ta + kCHeads, lo);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int hh = oct * 8 + j;
      if (hh < nh)
        asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst0 + int64_t(hh) * kLatent + mt * 128),
                     "f"((hi[j] + lo[j]) * sm.fac[hh])
                     : "memory");
    }
  }
  tc::tc_fence_before_sync();
  __syncthreads();
  tc::tc_fence_after_sync();
  if (wid == 0) tc::tmem_dealloc(tmem, kCTmemCols);
  // warp 1's (m, l) copies have read their shared source before the CTA exits
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ===========================================================================
// One CTA per (sequence, query, 32-head group) walking all the chunks: for
// large batches.  A cluster per head group puts S CTAs on S SMs for one
// head group, so a batch of 64 sequences x 2 head groups x 5 chunks needs
// about five rounds of the 28 clusters of 5 that fit at once; walking the
// chunks inside one CTA runs the 128 head groups side by side in one round.
// Per chunk: gather and dequantize the entries, S^T = KV . Q^T, softmax
// against a per-head reference maximum, O^T += V^T . P^T in tensor memory.
// The reference moves only when a chunk's maximum exceeds it by more than
// 2^8 (P stays below 256, which bf16 hi + lo and fp32 carry exactly enough);
// then the head's accumulated O and its sum are scaled by 2^(old - new)
// through tensor-memory loads and stores.  The output rows are written once,
// plainly (no zeroing, no reduce-adds).
// ===========================================================================
constexpr float kRescaleLog2 = 8.0f;

struct SeqSmall {
  uint64_t bar_s, bar_o;
  uint32_t valid[kCEntries / 32];                    // bit e: entry slot e holds an entry
  uint32_t tmem_slot;
  __align__(16) float red_m[4][4][8];                // [head octet][lane quarter][head]
  float red_l[4][4][8];
  float mref[kCHeads];                               // reference maximum (base 2), -inf: none yet
  float lsum[kCHeads];                               // sum of 2^(x - mref) over the entries so far
  int64_t rows[kMaxClusterSplits * kCEntries];       // cache row of every chunk's Top-K slot (-1: none)
};

size_t seq_smem_bytes() {
  return 1024 + size_t(kKvBytes) + size_t(kCQBytes) + size_t(2 * kCPRegion) + sizeof(SeqSmall);
}

// Cache rows of every chunk's Top-K slots (the checks of cluster_gather).
__device__ inline void seq_resolve_rows(const AttnArgs& a, int64_t* rows, int b, int S, int64_t n_ctx, int tid) {
  const int K = a.d.topk;
  for (int i = tid; i < S * kCEntries; i += kAttnThreads) {
    const int c = i / kCEntries, e = i % kCEntries;
    const int m0 = attn_chunk_main_lo(K, c, S), nm = attn_chunk_main_lo(K, c + 1, S) - m0;
    int64_t row = -1;
    if (e < nm) {
      const int32_t t = __ldg(a.topk + int64_t(b) * K + m0 + e);
      if (t >= 0 && t < n_ctx) {
        row = kv_row(a.page_table, a.d, b, t, a.ws);
        if (row < 0) row = -1;
      } else if (t >= n_ctx || t < -1) {
        raise_err(a.ws, CSA2_DEV_TOPK_IDX);
      }
    }
    rows[i] = row;
  }
}

// The reference maximum after a chunk whose maximum is mc, and the factor
// that rescales what was accumulated against the old one.
__device__ inline void seq_reference(float mo, float mc, float& mn, float& alpha) {
  mn = mo;
  if (mc != -INFINITY && (mo == -INFINITY || mc > mo + kRescaleLog2)) mn = mc;
  alpha = (mo == -INFINITY || mn == mo) ? 1.0f : exp2f(mo - mn);
}

__global__ void __launch_bounds__(kAttnThreads, 1) attn_seq_kernel(AttnArgs a, int early) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* kv_s = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);   // 9 x 16 KB
  uint8_t* q_s = kv_s + kKvBytes;                    // 9 x 4 KB: the query, kept for every chunk
  uint8_t* p_s = q_s + kCQBytes;                     // P^T hi / lo: two regions of 64 entries
  SeqSmall& sm = *reinterpret_cast<SeqSmall*>(p_s + 2 * kCPRegion);

  const int S = a.L.splits;
  const int nhg = (a.d.heads + kCHeads - 1) / kCHeads;
  const int qrow = blockIdx.x / nhg, hg = blockIdx.x % nhg;
  const int b = qrow / a.q_len, qi = qrow % a.q_len;
  const int H = a.d.heads, K = a.d.topk, W = a.d.swa;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool paged = a.page_table != nullptr;
  const int h0 = hg * kCHeads, nh = min(kCHeads, H - h0);
  if (wid == 0) tc::tmem_alloc(&sm.tmem_slot, kCTmemCols);
  if (tid == 0) {
    tc::mbar_init(&sm.bar_s, kSAcc);                 // one commit per S-issuing thread
    tc::mbar_init(&sm.bar_o, 4);                     // one commit per O-issuing thread
    tc::fence_mbar_init();
  }
  if (tid < kCHeads) {
    sm.mref[tid] = -INFINITY;
    sm.lsum[tid] = 0.0f;
  }
  {
    // L2 prefetch (hints: nothing is read into the SM) of what is read after
    // the wait: the query rows, the first chunk's window rows, the window length
    const char* qb = reinterpret_cast<const char*>(a.q + (int64_t(qrow) * H + h0) * kDqk);
    int w00, nw0;
    attn_chunk_window(K, W, 0, S, w00, nw0);
    const char* wb = reinterpret_cast<const char*>(a.swa + (int64_t(b) * W + w00) * kDqk);
    const int qlines = (nh * kDqk * 2 + 127) / 128, wlines = (nw0 * kDqk * 2 + 127) / 128;
    for (int i = tid; i < qlines + wlines; i += kAttnThreads) {
      const char* pf = i < qlines ? qb + 128 * i : wb + 128 * (i - qlines);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(pf));
    }
    if (tid == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.swa_len + b));
  }
  const int64_t n_ctx = checked_ctx(a.ctx_len, a.d, b, paged, a.ws);
  int m0 = attn_chunk_main_lo(K, 0, S), nm = attn_chunk_main_lo(K, 1, S) - m0, w0, nw;
  attn_chunk_window(K, W, 0, S, w0, nw);
  GatherCo g;
  if (early) {                                       // Reuse: the indices and the first chunk before the wait
    seq_resolve_rows(a, sm.rows, b, S, n_ctx, tid);
    __syncthreads();
    gather_load_co(a, g, sm.rows, nm, nw, wid, lane);
    gather_store_co(kv_s, g, wid, lane);
  }
  pdl_wait();
  pdl_launch_dependents();
  int swl = __ldg(a.swa_len + b);
  {
    constexpr int kQVec = kCHeads * (kDqk / 8);
    constexpr int kQPer = (kQVec + kAttnThreads - 1) / kAttnThreads;
    const uint4* qsrc = reinterpret_cast<const uint4*>(a.q + (int64_t(qrow) * H + h0) * kDqk);
    uint4 qv[kQPer];
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int i = tid + k * kAttnThreads;
      qv[k] = (i < kQVec && i / (kDqk / 8) < nh) ? __ldg(qsrc + i) : make_uint4(0, 0, 0, 0);
    }
    if (!early) {
      seq_resolve_rows(a, sm.rows, b, S, n_ctx, tid);
      __syncthreads();
      gather_load_co(a, g, sm.rows, nm, nw, wid, lane);
      gather_store_co(kv_s, g, wid, lane);
    }
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int i = tid + k * kAttnThreads;
      if (i < kQVec) {
        const int h = i / (kDqk / 8), j = i % (kDqk / 8);
        st_shared_v4(q_s, (j >> 3) * kCQRegion + tc::sw128_offset(h, j & 7), qv[k]);
      }
    }
  }
  if (swl < 0 || swl > W) {
    if (tid == 0 && hg == 0 && qi == 0) raise_err(a.ws, CSA2_DEV_SWA_LEN);
    swl = swl < 0 ? 0 : W;
  }
  swl = max(0, swl - (a.q_len - 1 - qi));            // the later queries' rows are not visible
  tc::tc_fence_before_sync();
  __syncthreads();
  tc::tc_fence_after_sync();
  const uint32_t tmem = sm.tmem_slot;
  const uint32_t kv_addr = tc::smem_u32(kv_s), q_addr = tc::smem_u32(q_s);
  const int quarter = wid & 3, oct = wid >> 2;       // lanes 32 quarter.., heads 8 oct..
  const int e = quarter * 32 + lane;
  const float c2 = a.scale * 1.4426950408889634f;    // logits in base 2
  bool ok = true;

  // the chunk's window rows are entries nm .. nm + nw - 1 (zeros at or past
  // swa_len); the first kWFirst 16-byte pieces a thread are loaded together
  // with the chunk's entries, at the end of the previous chunk's softmax
  constexpr int kWFirst = 4;
  uint4 wv[kWFirst];
  auto load_window_first = [&](int w0_, int nw_) {
    const uint4* src = reinterpret_cast<const uint4*>(a.swa + (int64_t(b) * W + w0_) * kDqk);
#pragma unroll
    for (int k = 0; k < kWFirst; ++k) {
      const int i = tid + k * kAttnThreads;
      wv[k] = (i < nw_ * (kDqk / 8) && w0_ + i / (kDqk / 8) < swl) ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
    }
  };
  load_window_first(w0, nw);
  for (int c = 0; c < S; ++c) {
    const int nwv = nw * (kDqk / 8);
    const uint4* wsrc = reinterpret_cast<const uint4*>(a.swa + (int64_t(b) * W + w0) * kDqk);
    if (c > 0) {
      // the previous chunk's O MMAs have read the tile and P^T
      ok = tc::mbar_wait_bounded(&sm.bar_o, uint32_t((c - 1) & 1)) && ok;
      tc::tc_fence_after_sync();
      gather_store_co(kv_s, g, wid, lane);
    }
#pragma unroll
    for (int k = 0; k < kWFirst; ++k) {
      const int i = tid + k * kAttnThreads;
      if (i < nwv) {
        const int r = i / (kDqk / 8), j = i % (kDqk / 8);
        st_shared_v4(kv_s, (j >> 3) * kRegion + tc::sw128_offset(nm + r, j & 7), wv[k]);
      }
    }
    for (int base = kWFirst * kAttnThreads; base < nwv; base += kWFirst * kAttnThreads) {
#pragma unroll
      for (int k = 0; k < kWFirst; ++k) {
        const int i = base + tid + k * kAttnThreads;
        wv[k] = (i < nwv && w0 + i / (kDqk / 8) < swl) ? __ldg(wsrc + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < kWFirst; ++k) {
        const int i = base + tid + k * kAttnThreads;
        if (i < nwv) {
          const int r = i / (kDqk / 8), j = i % (kDqk / 8);
          st_shared_v4(kv_s, (j >> 3) * kRegion + tc::sw128_offset(nm + r, j & 7), wv[k]);
        }
      }
    }
    {
      const int64_t* rows_c = sm.rows + c * kCEntries;
      const int ee = tid & (kCEntries - 1);
      const bool has = ee < nm ? rows_c[ee] >= 0 : (ee < nm + nw && w0 + ee - nm < swl);
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, has);
      if (tid < kCEntries && lane == 0) sm.valid[tid >> 5] = m;
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();

    // ---- S^T = KV . Q^T: 4 accumulators, 9 K steps spread over them ----------------------
    if (wid < kSAcc && lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16(kCEntries, kCHeads, 0, 0);
      const uint64_t ad0 = tc::smem_desc(kv_addr, 16, 1024, 2), bd0 = tc::smem_desc(q_addr, 16, 1024, 2);
      const int k4 = wid;
#pragma unroll
      for (int kb = 0; kb < 9; ++kb) {
        const uint32_t off = uint32_t(kb * kRegion + k4 * 32), qoff = uint32_t(kb * kCQRegion + k4 * 32);
        tc::mma_bf16(tmem + uint32_t(k4 * kCHeads), ad0 + (off >> 4), bd0 + (qoff >> 4), idS, kb > 0);
      }
      tc::mma_commit(&sm.bar_s);
    }
    __syncwarp();
    ok = tc::mbar_wait_bounded(&sm.bar_s, uint32_t(c & 1)) && ok;
    tc::tc_fence_after_sync();

    // ---- softmax against the reference maximum: 16 warps, 8 heads each -----------------
    float alpha[8];
    {
      float x[8];
      {
        const uint32_t ta = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(oct * 8);
        float x1[8], x2[8], x3[8];
        tc::tmem_ld8(ta, x);
        tc::tmem_ld8(ta + kCHeads, x1);
        tc::tmem_ld8(ta + 2 * kCHeads, x2);
        tc::tmem_ld8(ta + 3 * kCHeads, x3);
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = (x[j] + x1[j]) + (x2[j] + x3[j]);
      }
      const bool v_e = (sm.valid[e >> 5] >> (e & 31)) & 1;
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = v_e ? x[j] * c2 : -INFINITY;
      {
        float mx[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(mx[j]) : "f"(x[j]));
        if (lane == 0) {
          float4* dst = reinterpret_cast<float4*>(&sm.red_m[oct][quarter][0]);
          dst[0] = make_float4(mx[0], mx[1], mx[2], mx[3]);
          dst[1] = make_float4(mx[4], mx[5], mx[6], mx[7]);
        }
      }
      __syncthreads();
      float p[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float mc = fmaxf(fmaxf(sm.red_m[oct][0][j], sm.red_m[oct][1][j]),
                               fmaxf(sm.red_m[oct][2][j], sm.red_m[oct][3][j]));
        float mn;
        seq_reference(sm.mref[oct * 8 + j], mc, mn, alpha[j]);
        p[j] = (mn == -INFINITY || x[j] == -INFINITY) ? 0.0f : exp2f(x[j] - mn);
      }
      const float l = butterfly8<false>(p, lane);
      if ((lane & 3) == 0) sm.red_l[oct][quarter][octet_index(lane)] = l;
      uint8_t* reg = p_s + (e >> 6) * kCPRegion;
      const uint32_t ch = uint32_t((e >> 3) & 7), el = uint32_t(e & 7) * 2;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int h = oct * 8 + j;
        const uint32_t hb = pack_bf16x2(p[j], 0.0f);
        const float hv = __uint_as_float(hb << 16);
        *reinterpret_cast<uint16_t*>(reg + tc::sw128_offset(uint32_t(h), ch) + el) = uint16_t(hb & 0xFFFF);
        *reinterpret_cast<uint16_t*>(reg + tc::sw128_offset(uint32_t(kCHeads + h), ch) + el) =
            uint16_t(pack_bf16x2(p[j] - hv, 0.0f) & 0xFFFF);
      }
    }
    // ---- the heads whose reference moved: scale their accumulated O (the
    //      factors are the same in every lane of the warp) -----------------------------
    bool moved = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) moved = moved || alpha[j] != 1.0f;
    if (c > 0 && moved) {
#pragma unroll 1
      for (int mt = 0; mt < 4; ++mt) {
        const uint32_t ta = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(kCOCol + 64 * mt + oct * 8);
        float hi[8], lo[8];
        tc::tmem_ld8(ta, hi);
        tc::tmem_ld8(ta + kCHeads, lo);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          hi[j] *= alpha[j];
          lo[j] *= alpha[j];
        }
        tc::tmem_st8(ta, hi);
        tc::tmem_st8(ta + kCHeads, lo);
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();
    // the heads' running state (every thread has read the old reference), by
    // warp 1, while warps 0 and 2-4 issue the O MMAs
    if (wid == 1) {
      const int o8 = lane >> 3, j = lane & 7;
      const float mc = fmaxf(fmaxf(sm.red_m[o8][0][j], sm.red_m[o8][1][j]),
                             fmaxf(sm.red_m[o8][2][j], sm.red_m[o8][3][j]));
      float mn, al;
      seq_reference(sm.mref[lane], mc, mn, al);
      const float lc = (sm.red_l[o8][0][j] + sm.red_l[o8][1][j]) + (sm.red_l[o8][2][j] + sm.red_l[o8][3][j]);
      sm.lsum[lane] = sm.lsum[lane] * al + lc;
      sm.mref[lane] = mn;
    }
    // ---- O^T += V^T . [P_hi | P_lo]^T (4 M-tiles of 128 dims, N = 64, K = 128) ------------
    if ((wid == 0 || (wid >= 2 && wid <= 4)) && lane == 0) {
      constexpr uint32_t idO = tc::idesc_bf16(kCEntries, 2 * kCHeads, 1, 0);
      const uint64_t bp0 = tc::smem_desc(tc::smem_u32(p_s), 16, 1024, 2);
      const uint64_t av0 = tc::smem_desc(kv_addr, kRegion, 1024, 2);
      const int mt = wid == 0 ? 0 : wid - 1;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        tc::mma_bf16(tmem + kCOCol + 64 * mt, av0 + (((2 * mt) * kRegion + ks * 2048) >> 4),
                     bp0 + (((ks >> 2) * kCPRegion + (ks & 3) * 32) >> 4), idO, c > 0 || ks > 0);
      tc::mma_commit(&sm.bar_o);
    }
    __syncwarp();
    if (c + 1 < S) {                                 // the next chunk's entries and window: loads in flight
      m0 = attn_chunk_main_lo(K, c + 1, S);
      nm = attn_chunk_main_lo(K, c + 2, S) - m0;
      attn_chunk_window(K, W, c + 1, S, w0, nw);
      load_window_first(w0, nw);
      gather_load_co(a, g, sm.rows + (c + 1) * kCEntries, nm, nw, wid, lane);
    }
  }
  ok = tc::mbar_wait_bounded(&sm.bar_o, uint32_t((S - 1) & 1)) && ok;
  tc::tc_fence_after_sync();
  __syncthreads();
  if (!ok && tid == 0) raise_err(a.ws, CSA2_DEV_TIMEOUT);
  // ---- out = O / sum, lse = ref ln 2 + ln(sum): a warp's 32 lanes write 32
  //      consecutive dims of one head ----------------------------------------------------
  float* dst0 = a.out + (int64_t(qrow) * H + h0) * kLatent + quarter * 32 + lane;
#pragma unroll 1
  for (int mt = 0; mt < 4; ++mt) {
    float hi[8], lo[8];
    const uint32_t ta = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(kCOCol + 64 * mt + oct * 8);
    tc::tmem_ld8(ta, hi);
    tc::tmem_ld8(ta + kCHeads, lo);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int hh = oct * 8 + j;
      if (hh < nh) {
        const float L = sm.lsum[hh];
        dst0[int64_t(hh) * kLatent + mt * 128] = L > 0.0f ? (hi[j] + lo[j]) / L : 0.0f;
      }
    }
  }
  if (tid < nh) {
    const float L = sm.lsum[tid];
    a.lse[int64_t(qrow) * H + h0 + tid] = L > 0.0f ? sm.mref[tid] * 0.6931471805599453f + logf(L) : -INFINITY;
  }
  tc::tc_fence_before_sync();
  __syncthreads();
  tc::tc_fence_after_sync();
  if (wid == 0) tc::tmem_dealloc(tmem, kCTmemCols);
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

// Clusters of `chunks` attention CTAs that fit on the device at once (read
// once per device and cluster size).
static int cluster_capacity(int chunks, size_t smem) {
  static std::atomic<int> cap[kMaxDevices][kMaxClusterSplits + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  int n = cap[dev][chunks].load(std::memory_order_relaxed);
  if (n > 0) return n;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = unsigned(chunks);
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.gridDim = dim3(unsigned(chunks), 1, 1);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&n, attn_cluster_kernel, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = max(1, device_sms() / chunks);               // no answer: as if every SM took a CTA
  }
  cap[dev][chunks].store(n, std::memory_order_relaxed);
  return n;
}

// Whether the chunk-walking kernel finishes before the clusters: rounds of
// clusters (about 13 us each: gather, S, softmax, merge) against rounds of
// one CTA per head group that sets up in about 6 us and walks `chunks`
// chunks at about 7.5 us each -- figures measured on this GPU (128K,
// 4-query and serving-mix workloads; tenths of a microsecond below).
static bool attention_walks_chunks(int items, int chunks, size_t cluster_smem) {
  const int cap = cluster_capacity(chunks, cluster_smem);
  const int64_t cluster_rounds = (items + cap - 1) / cap;
  const int64_t seq_rounds = (items + device_sms() - 1) / device_sms();
  return seq_rounds * (60 + 75 * int64_t(chunks)) < cluster_rounds * 130;
}

cudaError_t launch_attention(AttnArgs a, cudaStream_t st) {
  const int H = a.d.heads, K = a.d.topk, W = a.d.swa;
  if (!attn_uses_partials(a.d)) {
    // one cluster of 128-entry chunks per (sequence, group of 32 heads), or,
    // for many head groups, one CTA per head group walking the chunks
    const int chunks = a.L.splits;
    const int nhg = (H + kCHeads - 1) / kCHeads;
    const size_t smem = cluster_smem_bytes();
    static KernelAttrs done;
    cudaError_t e = prepare_kernel(attn_cluster_kernel, smem, false, done);
    if (e != cudaSuccess) return e;
    const int items = nhg * a.batch * a.q_len;
    if (attention_walks_chunks(items, chunks, smem)) {
      const size_t sm2 = seq_smem_bytes();
      static KernelAttrs done_seq;
      e = prepare_kernel(attn_seq_kernel, sm2, false, done_seq);
      if (e != cudaSuccess) return e;
      CSA2_PROFILED(st, "attn_seq_tc",
                    (e = launch_pdl(attn_seq_kernel, dim3(unsigned(items)), dim3(kAttnThreads), sm2, st, 1, a,
                                    a.early)));
      return e;
    }
    CSA2_PROFILED(st, "attn_cluster_tc",
                  (e = launch_pdl(attn_cluster_kernel, dim3(unsigned(chunks), unsigned(nhg * a.batch * a.q_len), 1),
                                  dim3(kAttnThreads), smem, st, unsigned(chunks), a, a.early)));
    return e;
  }
  // more than 8 chunks: one CTA per 128-entry chunk writes partials,
  // the combine kernel merges them
  CUtensorMap qmap, swamap;
  if (!encode_rows_map(&qmap, a.q, uint64_t(a.batch) * H, kQRows)) return cudaErrorInvalidValue;
  // the window is loaded by TMA when it starts a 128-entry split
  int swa_split = -1;
  if (W > 0 && W <= kEntries && K % kEntries == 0) swa_split = K / kEntries;
  swamap = qmap;
  if (swa_split >= 0 && !encode_rows_map(&swamap, a.swa, uint64_t(a.batch) * W, kEntries))
    return cudaErrorInvalidValue;
  const size_t smem = attn_smem_bytes(H);
  static KernelAttrs done_partial;
  cudaError_t e = prepare_kernel(attn_partial_tc_kernel, smem, false, done_partial);
  if (e != cudaSuccess) return e;
  CSA2_PROFILED(st, "attn_partial_tc",
                (e = launch_pdl(attn_partial_tc_kernel, dim3(unsigned(a.L.splits), unsigned(a.batch)),
                                dim3(kAttnThreads), smem, st, 1, a, qmap, swamap, swa_split)));
  if (e != cudaSuccess) return e;
  CSA2_PROFILED(st, "attn_combine", (e = launch_pdl(attn_combine_kernel, dim3(unsigned(H), unsigned(a.batch)),
                                                    dim3(128), 0, st, 1, a)));
  return e;
}

}  // namespace csa2
