// scan_fp4.cu -- indexer scan with FP4 query and keys on the tcgen05 tensor
// cores (Full: every visible position; Reindex: the pool positions).
//
// Format (foosynaptic atlas "DeepSeek-V4.1-Flash 梗概", section 3.2, "FP4 main
// KV"; the indexer's query and key were trained for FP4, newsaint.id
// "DeepSeek-V4.1-Flash 2026: ...", section 4): E2M1 values with one E4M3
// scale per 16 channels; the score is that of the dequantized values,
//   d_{t,h} = sum_g sk_{t,g} sq_{h,g} D_{t,h,g},  D_{t,h,g} = sum_{c in g} qhat_{h,c} khat_{t,c},
//   s_t = sum_h w_h ReLU(d_{t,h}).
//
// Exact group dots on the tensor cores.  Every E2M1 level times 2 is an
// integer, so D is a multiple of 1/4 with |D| <= 16 * 36 = 576.  The keys and
// the query are widened to E4M3 bytes worth 2^-6 times their E2M1 values (a
// bit shuffle, exact; within every 8 channels the even ones first, the same in
// keys and query) and multiplied with kind::f8f6f4: every product is a
// multiple of 2^-14 below 2^-6 * 36 and every partial sum a multiple of 2^-14
// below 2^-3, so the tensor core forms D * 2^-12 without any rounding (the
// accumulation keeps far more than the 12 bits involved).  One MMA per 32
// channels (two groups) with N = 32: B row (p, h) holds the query of head h
// in the groups of parity p and zeros elsewhere, so column 32 ks + 16 p + h
// of the k-step's accumulator is D_{t,h,2ks+p}: 128 columns per tile, one per
// (group, head).
//
// Scales and the bound in fp32 (pairs of heads per f32x2 instruction, each
// lane rounded as a scalar one).  y = (sk * 4096) * D2 (D2 = the accumulator)
// is exact (<= 16 significant bits); d_h = sum_g sq_{h,g} y_g is a chain of 8
// FMAs (7 roundings) and v = sum_h w_h max(d_h, 0) a chain of 16 FMAs, so
//   |v - s| <= (gamma_7 + gamma_16 (1 + gamma_7)) sum_h |w_h| sum_c |q_hc k_tc|
// (plus the fp64 rounding of the exact score), a bound that holds for any
// tensor-core accumulation order.  With |khat| <= 6 the last sum is at most
//   6 sum_g sk_{t,g} U_g,   U_g = sum_h |w_h| sq_{h,g} sum_{c in g} |qhat_{h,c}|,
// so delta_t = sum_g sk_{t,g} ub_g with ub_g = coef * 6 * U_g, all rounded
// upwards, plus 2^-140 for a possible underflow of w_h * ReLU(d_h).
//
// Work: one persistent CTA per SM over a contiguous range of 128-position
// tiles, roles in warps handing tiles on through mbarriers:
//   * warp 0: TMA of the tile's FP4 codes (64 B per row) into an 8-stage ring
//     (Reindex: one 8-row box per pool block);
//   * warps 2-5 (converter): the query of a new sequence is quantized and laid
//     out as B; each tile's codes become 128-byte swizzled K-major E4M3 rows
//     in one of 4 operand stages, followed by a copy of B;
//   * warp 1 (one thread): 4 MMAs per tile (M = 128, N = 32, K = 32) into one
//     of four tensor-memory accumulators;
//   * warps 6-9, 10-13, 14-17 (three epilogue groups, tiles in turn): the
//     row's 8 key scales (read from global memory two of the group's tiles
//     ahead), scores, bound, block maxima, writes.  The epilogue is the
//     slowest role, so three groups work on three tiles at once.
#include <cmath>

#include "common.cuh"
#include "fp4.cuh"
#include "kernels.cuh"
#include "profile.cuh"
#include "scan_common.cuh"
#include "tc.cuh"

namespace csa2 {

namespace {

constexpr int kConvWarps = 4;             // converter warps 2-5, four code rows per thread
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kEpiWarp0 = 2 + kConvWarps;  // epilogue groups from warp 6, four warps each
constexpr int kEpiGroups = 3;             // tile k goes to group k % 3
constexpr int kEpiThreads = 128;          // threads of an epilogue group: one per row
constexpr int kFThreads = 32 * (kEpiWarp0 + 4 * kEpiGroups);
constexpr int kCStages = 8;               // code ring depth
constexpr int kCodeBytes = kTile * 64;    // 8 KB of FP4 codes per tile
constexpr int kAStages = 4;               // operand stages
constexpr int kAKeyBytes = kTile * 128;   // 16 KB of widened keys
constexpr int kBBytes = 32 * 128;         // B: 32 rows of 128 channels
constexpr int kAStride = kAKeyBytes + kBBytes;
constexpr int kDBufs = kEpiGroups + 1;
constexpr int kDCols = 128;               // accumulator columns per tile
static_assert(kDBufs * kDCols <= 512, "accumulators fit in tensor memory");
constexpr uint32_t kTmemCols = 512;

struct FScanSmem {
  uint8_t astage[kAStages][kAStride];     // widened keys, then B; 1024-aligned
  uint8_t craw[kCStages][kCodeBytes];     // FP4 codes as loaded
  uint8_t qb[kBBytes];                    // the converter's current B
  float sq[kEpiGroups][8][kMaxIdxHeads];  // [epilogue group][group g][head h]: query scale
  float wv[kEpiGroups][kMaxIdxHeads];     // [epilogue group]: w_h (0 past the heads)
  float ub[kEpiGroups][8];                // [epilogue group]: bound factor per key group
  float ucon[kEpiGroups][8][kMaxIdxHeads];  // [epilogue group]: |w_h| sq_hg sum|qhat|, rounded up
  int64_t seq_items[kSeqCache];
  int32_t n_seq_cached;
  uint64_t cfull[kCStages], cempty[kCStages];
  uint64_t afull[kAStages], aempty[kAStages];
  uint64_t d_full[kDBufs], d_empty[kDBufs];
  uint32_t tmem_slot;
  volatile int32_t abort_flag;
};

// The query of head h, group g (16 bf16 channels) of sequence b, quantized:
// 8 bytes of codes and the scale code.  Heads past hi quantize zeros.
__device__ inline uint2 query_group(const IdxArgs& a, int b, int h, int g, uint32_t* sc) {
  uint4 lo = make_uint4(0, 0, 0, 0), hi4 = make_uint4(0, 0, 0, 0);
  if (h < a.d.idx_heads) {
    const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.idx_q) +
                                                      (int64_t(b) * a.d.idx_heads + h) * 128 + 16 * g);
    lo = __ldg(src);
    hi4 = __ldg(src + 1);
  }
  return fp4_quantize_group(lo, hi4, sc);
}

__device__ inline void conv_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConvThreads) : "memory");
}

// Converter group (gt = 0..127 owns head gt/8, group gt%8): B of sequence b
// into sm.qb.  Row 16 p + h holds the widened query of head h in the groups of
// parity p; the chunks of the other parity are zero.  So column 32 ks + 16 p
// + h of a tile's accumulator is head h's dot over group 2 ks + p: column
// 16 g + h for group g.
__device__ void build_b(const IdxArgs& a, FScanSmem& sm, int b, int gt) {
  const int h = (gt >> 3) & 15, g = gt & 7;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (gt < 128) {
    uint32_t sc;
    const uint2 c = query_group(a, b, h, g, &sc);
    e2m1x8_to_e4m3x8_scaled(c.x, v.x, v.y);
    e2m1x8_to_e4m3x8_scaled(c.y, v.z, v.w);
  }
  conv_sync();                                     // the previous B has been copied out
  if (gt < 128) {
    const int p = g & 1;
    *reinterpret_cast<uint4*>(sm.qb + tc::sw128_offset(16 * p + h, g)) = v;
    *reinterpret_cast<uint4*>(sm.qb + tc::sw128_offset(16 * (1 - p) + h, g)) = make_uint4(0, 0, 0, 0);
  }
  conv_sync();
}

__device__ inline void epi_sync(int eg) {
  asm volatile("bar.sync %0, %1;" ::"r"(2 + eg), "n"(kEpiThreads) : "memory");
}

// Epilogue group eg (gt = 0..127 owns head gt/8, group gt%8): the scales,
// weights and bound factors of sequence b.
__device__ void epi_query(const IdxArgs& a, FScanSmem& sm, int b, int gt, int eg) {
  const int h = (gt >> 3) & 15, g = gt & 7, hi = a.d.idx_heads;
  const bool own = gt < 128;
  uint32_t sc = 0;
  uint2 c = make_uint2(0, 0);
  if (own) c = query_group(a, b, h, g, &sc);
  const float wh = own && h < hi ? __ldg(a.w + int64_t(b) * hi + h) : 0.0f;
  const float wg = gt < hi ? __ldg(a.w + int64_t(b) * hi + gt) : 0.0f;
  // 2 * sum |qhat| over the group: twice each level is an integer
  const uint32_t twice[4] = {e2m1x4_to_i8x4_twice(c.x & 0x7777u), e2m1x4_to_i8x4_twice((c.x >> 16) & 0x7777u),
                             e2m1x4_to_i8x4_twice(c.y & 0x7777u), e2m1x4_to_i8x4_twice((c.y >> 16) & 0x7777u)};
  int s2 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) s2 = __dp4a(int(twice[i]), int(0x01010101), s2);
  const float sqv = own && h < hi ? e4m3_to_f32(sc) : 0.0f;
  epi_sync(eg);                                    // the previous sequence's values are no longer read
  if (own) {
    sm.sq[eg][g][h] = sqv;
    sm.ucon[eg][g][h] = __fmul_ru(fabsf(wh), sqv * float(s2) * 0.5f);   // sqv * s2 / 2 is exact
  }
  if (gt < kMaxIdxHeads) sm.wv[eg][gt] = wg;
  epi_sync(eg);
  if (gt < 8) {
    float u = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxIdxHeads; ++i) u = __fadd_ru(u, sm.ucon[eg][gt][i]);
    sm.ub[eg][gt] = __fmul_ru(__fmul_ru(a.err_coef, 6.0f), u);
  }
  epi_sync(eg);
}

// Packed pairs of fp32 values (two heads) for the f32x2 instructions: each
// lane of a pair is rounded exactly as the scalar instruction would round it.
__device__ inline uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ inline void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ inline uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ inline uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// d_h += sq_{h,g} * (sk'_g * D2[16 (g - g0) + h]) over the 2 groups g0, g0+1,
// two heads per instruction (acc2[j] holds heads 2j, 2j+1).
__device__ inline void group_terms(const FScanSmem& sm, int eg, int g0, const float (&dv)[32], const float (&skp)[8],
                                   uint64_t (&acc2)[kMaxIdxHeads / 2]) {
#pragma unroll
  for (int gg = 0; gg < 2; ++gg) {
    const int g = g0 + gg;
    const uint64_t sk2 = f2_pack(skp[g], skp[g]);
    const ulonglong2* sq2 = reinterpret_cast<const ulonglong2*>(sm.sq[eg][g]);
#pragma unroll
    for (int j4 = 0; j4 < 4; ++j4) {
      const ulonglong2 s = sq2[j4];                       // heads 4 j4 .. 4 j4 + 3
      const int c = 16 * gg + 4 * j4;
      const uint64_t y0 = f2_mul(sk2, f2_pack(dv[c], dv[c + 1]));        // exact
      const uint64_t y1 = f2_mul(sk2, f2_pack(dv[c + 2], dv[c + 3]));
      acc2[2 * j4] = f2_fma(s.x, y0, acc2[2 * j4]);
      acc2[2 * j4 + 1] = f2_fma(s.y, y1, acc2[2 * j4 + 1]);
    }
  }
}

// Epilogue of one tile for the thread owning row r (TMEM lanes of warp
// quarter r / 32) of epilogue group eg.
__device__ inline void fp4_epilogue(const IdxArgs& a, bool reindex, const FScanSmem& sm, int eg, const TileRef& pt,
                                    uint32_t tmem_d, int64_t row, uint2 kscale, int r, int lane) {
  float skp[8], sk[8];
  const uint32_t kw[2] = {kscale.x, kscale.y};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t h2 = e4m3x2_to_f16x2(uint16_t(kw[i >> 1] >> (16 * (i & 1))));
    sk[2 * i] = __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFF)));
    sk[2 * i + 1] = __half2float(__ushort_as_half(uint16_t(h2 >> 16)));
  }
#pragma unroll
  for (int g = 0; g < 8; ++g) skp[g] = sk[g] * 4096.0f;    // undoes the 2^-6 * 2^-6 of the widening
  uint64_t acc2[kMaxIdxHeads / 2];
#pragma unroll
  for (int j = 0; j < kMaxIdxHeads / 2; ++j) acc2[j] = 0;
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {                          // groups 2ks, 2ks+1
    float dv[32];
    tc::tmem_ld32(tmem_d + 32 * ks, dv);
    group_terms(sm, eg, 2 * ks, dv, skp, acc2);
  }
  float v = 0.0f;
#pragma unroll
  for (int j = 0; j < kMaxIdxHeads / 2; ++j) {
    float d0, d1;
    f2_unpack(acc2[j], d0, d1);
    v = __fmaf_rn(sm.wv[eg][2 * j], fmaxf(d0, 0.0f), v);
    v = __fmaf_rn(sm.wv[eg][2 * j + 1], fmaxf(d1, 0.0f), v);
  }
  float delta = 0x1p-140f;
#pragma unroll
  for (int g = 0; g < 8; ++g) delta = __fmaf_ru(sk[g], sm.ub[eg][g], delta);
  const bool valid = row >= 0;
  if (!valid) { v = -INFINITY; delta = 0.0f; }
  float bmax = v, bd = delta;
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    bmax = fmaxf(bmax, __shfl_xor_sync(0xFFFFFFFFu, bmax, o));
    bd = fmaxf(bd, __shfl_xor_sync(0xFFFFFFFFu, bd, o));
  }
  float* ws_f = reinterpret_cast<float*>(a.ws);
  const int64_t t = pt.t0 + r;
  if (reindex) {
    const int64_t P8 = int64_t(a.d.pool_blocks) * kBlock;
    if (r < pt.nvalid) ws_f[(a.L.ri_scores >> 2) + int64_t(pt.b) * P8 + t] = v;
    if ((lane & 7) == 0 && r < pt.nvalid)
      ws_f[(a.L.ri_delta >> 2) + int64_t(pt.b) * a.d.pool_blocks + (t >> 3)] = bd;
    return;
  }
  if (valid) ws_f[(a.L.pos_scores >> 2) + int64_t(pt.b) * a.d.max_ctx + t] = v;
  if ((lane & 7) == 0 && r < pt.nvalid) {
    const int64_t j = t >> 3;
    ws_f[(a.L.blk_scores >> 2) + int64_t(pt.b) * a.L.nb_max + j] = bmax;
    ws_f[(a.L.blk_delta >> 2) + int64_t(pt.b) * a.L.nb_max + j] = bd;
  }
}

__global__ void __launch_bounds__(kFThreads, 1)
    scan_fp4_kernel(IdxArgs a, const __grid_constant__ CUtensorMap kmap, bool reindex) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  FScanSmem& sm = *reinterpret_cast<FScanSmem*>(smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  __shared__ int64_t total_tiles_s;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // early inputs: the lengths and the keys may be read before the previous
  // kernel finishes; everything else waits for it (below)
  if (!a.early) {
    pdl_wait();
    pdl_launch_dependents();
  }
  if (wid == 0) {
    const int64_t tsum = count_tiles(a, sm, reindex, lane);
    if (lane == 0) total_tiles_s = tsum;
  }
  __syncthreads();
  const int64_t T = total_tiles_s;
  const int64_t g0 = int64_t(blockIdx.x) * T / gridDim.x;
  const int64_t g1 = int64_t(blockIdx.x + 1) * T / gridDim.x;
  if (g0 >= g1) return;

  if (wid == 0) tc::tmem_alloc(&sm.tmem_slot, kTmemCols);
  if (tid == 0) {
    for (int s = 0; s < kCStages; ++s) {
      tc::mbar_init(&sm.cfull[s], 1);             // the producer's arrival (with its TMA bytes)
      tc::mbar_init(&sm.cempty[s], kConvWarps);   // the converter warps
    }
    for (int s = 0; s < kAStages; ++s) {
      tc::mbar_init(&sm.afull[s], kConvWarps);    // the converter warps
      tc::mbar_init(&sm.aempty[s], 1);            // the MMAs' commit
    }
    for (int i = 0; i < kDBufs; ++i) {
      tc::mbar_init(&sm.d_full[i], 1);
      tc::mbar_init(&sm.d_empty[i], 4);           // the 4 warps of an epilogue group
    }
    tc::fence_mbar_init();
    sm.abort_flag = 0;
  }
  tc::tc_fence_before_sync();
  __syncthreads();
  tc::tc_fence_after_sync();
  const uint32_t tmem = sm.tmem_slot;
  const int ntiles = int(g1 - g0);
  if (a.early && wid != 0) {
    // the producer (warp 0) waits once its first ring of codes is in flight
    pdl_wait();
    pdl_launch_dependents();
  }

  if (wid == 0) {
    // ================= producer: FP4 codes =================
    if (reindex)
      produce_reindex<64, kCStages>(a, &kmap, sm, sm.craw[0], kCodeBytes, sm.cfull, sm.cempty, g0, ntiles, lane,
                                    a.early != 0);
    else if (lane == 0)
      produce_full<64, kCStages>(a, &kmap, sm, sm.craw[0], kCodeBytes, sm.cfull, sm.cempty, g0, ntiles,
                                 a.early != 0);
  } else if (wid == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3(kTile, 32);
      const uint64_t a0 = tc::smem_desc(tc::smem_u32(sm.astage[0]), 16, 1024, 2);
      const uint64_t b0 = tc::smem_desc(tc::smem_u32(sm.astage[0] + kAKeyBytes), 16, 1024, 2);
      int issued = 0;
      RingPos<kAStages> ring;
      for (int k = 0; k < ntiles; ++k, ring.next()) {
        const int buf = k % kDBufs;
        if (!wait_or_abort(sm, &sm.afull[ring.stage], ring.phase)) break;
        if (k >= kDBufs && !wait_or_abort(sm, &sm.d_empty[buf], uint32_t((k / kDBufs - 1) & 1))) break;
        tc::tc_fence_after_sync();
        const uint64_t off = uint64_t(ring.stage) * (kAStride >> 4);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)                 // 32 channels = 32 bytes per k-step
          mma_f8(tmem + kDCols * buf + 32 * ks, a0 + off + 2 * ks, b0 + off + 2 * ks, idesc, false);
        tc::mma_commit(&sm.aempty[ring.stage]);
        tc::mma_commit(&sm.d_full[buf]);
        issued = k + 1;
      }
      // after an abort, let the issued MMAs finish before the tensor memory is freed
      if (sm.abort_flag && issued > 0)
        tc::mbar_wait_bounded(&sm.d_full[(issued - 1) % kDBufs], uint32_t(((issued - 1) / kDBufs) & 1),
                              20ull * 1000 * 1000);
    }
  } else if (wid < kEpiWarp0) {
    // ================= converter (warps 2-5) =================
    const int gt = tid - 64;
    const int j = gt & 3;                              // 16-byte piece of a code row: channels 32j .. 32j+31
    int cb = 0, cur_b = -1;
    int64_t cbase = 0;
    RingPos<kCStages> cring;
    RingPos<kAStages> aring;
    for (int k = 0; k < ntiles; ++k, cring.next(), aring.next()) {
      const TileRef tr = tile_of(a, sm, reindex, g0 + k, cb, cbase);
      if (tr.b != cur_b) {
        build_b(a, sm, tr.b, gt);
        cur_b = tr.b;
      }
      if (!wait_or_abort(sm, &sm.cfull[cring.stage], cring.phase)) break;
      if (k >= kAStages && !wait_or_abort(sm, &sm.aempty[aring.stage], aring.phase ^ 1u)) break;
      const uint8_t* src = sm.craw[cring.stage];
      uint8_t* dst = sm.astage[aring.stage];
      uint4 cw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) cw[i] = *reinterpret_cast<const uint4*>(src + ((gt >> 2) + 32 * i) * 64 + 16 * j);
      __syncwarp();
      if (lane == 0) arrive(&sm.cempty[cring.stage]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t r = uint32_t((gt >> 2) + 32 * i);
        const uint32_t w[4] = {cw[i].x, cw[i].y, cw[i].z, cw[i].w};
        uint32_t e[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) e2m1x8_to_e4m3x8_scaled(w[u], e[2 * u], e[2 * u + 1]);
        *reinterpret_cast<uint4*>(dst + tc::sw128_offset(r, 2 * j)) = make_uint4(e[0], e[1], e[2], e[3]);
        *reinterpret_cast<uint4*>(dst + tc::sw128_offset(r, 2 * j + 1)) = make_uint4(e[4], e[5], e[6], e[7]);
      }
#pragma unroll
      for (int i = 0; i < kBBytes / 16 / kConvThreads; ++i)
        reinterpret_cast<uint4*>(dst + kAKeyBytes)[gt + i * kConvThreads] =
            reinterpret_cast<const uint4*>(sm.qb)[gt + i * kConvThreads];
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) arrive(&sm.afull[aring.stage]);
    }
  } else {
    // ================= epilogue groups (four warps each, tiles in turn) ==========
    const int eg = (wid - kEpiWarp0) >> 2;
    const int gt = tid - 32 * kEpiWarp0 - eg * kEpiThreads;
    const int quarter = wid & 3;                       // TMEM lanes 32*quarter ..
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    // the row's cache row and key scales are loaded two of the group's tiles
    // ahead, so that their memory latency overlaps the tiles in between
    int pb = 0, cur_b = -1;
    int64_t pbase = 0;
    TileRef tA = {0, 0, 0}, tB = {0, 0, 0};
    int64_t rA = -1, rB = -1;
    uint2 kA = make_uint2(0, 0), kB = make_uint2(0, 0);
    auto fetch = [&](int kk, TileRef& t, int64_t& row, uint2& ks) {
      if (kk >= ntiles) return;
      t = tile_of(a, sm, reindex, g0 + kk, pb, pbase);
      row = row_of(a, reindex, t, r);
      ks = row >= 0 ? __ldg(reinterpret_cast<const uint2*>(a.idx_scales + row * 8)) : make_uint2(0, 0);
    };
    fetch(eg, tA, rA, kA);
    fetch(eg + kEpiGroups, tB, rB, kB);
    for (int k = eg; k < ntiles; k += kEpiGroups) {
      const TileRef tr = tA;
      const int64_t row = rA;
      const uint2 ks = kA;
      tA = tB;
      rA = rB;
      kA = kB;
      fetch(k + 2 * kEpiGroups, tB, rB, kB);
      if (tr.b != cur_b) {
        epi_query(a, sm, tr.b, gt, eg);
        cur_b = tr.b;
      }
      const int buf = k % kDBufs;
      if (!wait_or_abort(sm, &sm.d_full[buf], uint32_t((k / kDBufs) & 1))) break;
      tc::tc_fence_after_sync();
      fp4_epilogue(a, reindex, sm, eg, tr, tmem + lane_base + kDCols * buf, row, ks, r, lane);
      tc::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) arrive(&sm.d_empty[buf]);
    }
  }
  tc::tc_fence_before_sync();
  __syncthreads();
  if (sm.abort_flag && tid == 0) raise_err(a.ws, CSA2_DEV_TIMEOUT);
  if (wid == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

double gamma_n(int n, double u) { return n * u / (1.0 - n * u); }

// coef: the fp32 FMA chains of the group sum (8 terms) and of the head sum
// (up to 16 terms), and the fp64 rounding of the exact score, relative to
// sum_h |w_h| sum_c |q_hc k_tc|.
float fp4_err_coef() {
  const double u32 = std::ldexp(1.0, -24), u64 = std::ldexp(1.0, -53);
  const double g7 = gamma_n(7, u32), g16 = gamma_n(kMaxIdxHeads, u32), g64 = gamma_n(kMaxIdxHeads + 2, u64);
  return float((g7 + g16 * (1.0 + g7) + g64) * 1.01);
}

}  // namespace

cudaError_t launch_scan_fp4(const IdxArgs& args, bool reindex, cudaStream_t st) {
  IdxArgs a = args;
  a.err_coef = fp4_err_coef();
  CUtensorMap map;
  cudaError_t e = idx_key_map(&map, a, reindex, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  const int64_t grid = scan_grid(a, reindex);
  const size_t smem = sizeof(FScanSmem) + 1024;
  static KernelAttrs done;
  e = prepare_kernel(scan_fp4_kernel, smem, false, done);
  if (e != cudaSuccess) return e;
  CSA2_PROFILED(st, reindex ? "reindex_score_fp4" : "indexer_scan_fp4",
                (e = launch_pdl(scan_fp4_kernel, dim3(unsigned(grid)), dim3(kFThreads), smem, st, 1, a, map,
                                reindex)));
  return e;
}

}  // namespace csa2
