// scan.cu -- Full-mode indexer scan on the tcgen05 tensor cores (E4M3 keys).
//
// For every visible position t (foosynaptic atlas "DeepSeek-V4.1-Flash 梗概",
// section 3.2: the first Full layer scores every causally visible position):
//   d_{t,h} = q_h . k_t,  s_t = sum_h w_h ReLU(d_{t,h}),  bs_j = max over block j,
// and a rigorous bound delta_j >= |s_t - v_t| for the approximate v_t.
//
// The MMAs take the E4M3 keys exactly as they sit in the cache
// (kind::f8f6f4, E4M3 x E4M3, fp32 accumulation in tensor memory); nothing
// converts them.  The bf16 query is split exactly into two E4M3 pieces per
// head, Qs = q_h 2^e_h = q1 + r1 (e_h puts max |q_h| 2^e_h in [2^7, 2^8); q1 is
// the E4M3 rounding of Qs and r1 the remainder, which has at most 4
// significant bits and is exact in E4M3 unless it falls below 2^-9 -- that
// rare loss is counted in the bound).
//
// Work: one persistent CTA per SM walks a contiguous range of 128-position
// tiles; its warps specialise and hand tiles on through mbarriers, so the
// key stream, the MMAs and the epilogue of consecutive tiles overlap.  Each
// stage of the 10-stage shared-memory ring holds a tile's keys (128 rows x
// 128 B, 128-byte swizzled K-major) followed by the query pieces (32 rows:
// q1 of the 16 heads, then r1), so that one MMA per K-step with A = the keys
// and B = the whole stage (N = 160) yields, per position t,
//   columns 0..127:   the Gram row k_t . k_s  (its diagonal is ||k_t||^2),
//   columns 128..159: k_t . q1_h and k_t . r1_h.
//   * warp 0: one thread streams the keys of each tile by TMA (tensor map
//     with the same swizzle); for Reindex tiles (16 scattered pool blocks)
//     the warp resolves the rows of a window of up to 10 tiles at a time and
//     16 lanes load a tile's blocks with one 8-row TMA box each.
//   * warps 2-5 (the query group) split the query when a new sequence starts
//     and copy the pieces into each stage behind its keys.
//   * warp 1 (one thread) issues the 4 MMAs of a tile (kind::f8f6f4, M=128,
//     N=160, K=32 each) into the next of three tensor-memory accumulators.
//   * warps 6-9 and 10-13, two epilogue groups taking alternate tiles from
//     three tensor-memory accumulators: v_t = sum_h w'_h ReLU(D_h + D_{16+h}) with
//     w'_h = w_h 2^-e_h, block max over 8 positions, and the bound
//       delta_t = C ||u||_2 ||k_t||_2 + (query rounding term),
//     u_c = sum_h |w'_h| (|q1_hc| + |r1_hc|): by Cauchy-Schwarz it is at least
//     C sum_c u_c |k_tc|, which covers the error of the weighted head sum.
// C covers the tensor-core accumulation.  The model: within one MMA step the
// 32 products are aligned to the largest of them and kept to 2^-23 of it
// (at most 2^-18 of the step's sum|products|), and the 3 additions of step
// results into the fp32 accumulator round to nearest (2^-24 each): at most
// 2^-17.8 of sum|products| per dot product.  C takes 2^-16, a margin of 3.5
// over the model; the worst observed on adversarial operands (one dominant
// product per step, the others small, same-signed, just below a power of
// two) is 2^-18.8, and products are not re-aligned against a large running
// sum (the later steps of that test lose nothing).  C also covers the fp32
// head sum and the fp64 rounding of the exact score.  ||k_t||^2 comes from the
// same MMA (all its products are positive, so it is low by at most 2^-14 of
// itself) and is raised accordingly before the square root.
#include <cmath>

#include "common.cuh"
#include "kernels.cuh"
#include "profile.cuh"
#include "scan_common.cuh"
#include "tc.cuh"

namespace csa2 {

constexpr int kScanThreads = 448;          // warp 0 TMA, 1 MMA, 2-5 query, 6-9 / 10-13 epilogue
constexpr int kStages = 10;                // ring depth
constexpr int kKeyBytes = kTile * 128;     // 16 KB of E4M3 keys
constexpr int kQpBytes = 32 * 128;         // q1 (16 rows) + r1 (16 rows)
constexpr int kStageStride = kKeyBytes + kQpBytes;
constexpr int kMmaN = kTile + 32;          // Gram row + the two query pieces
constexpr int kDBufs = 3;                  // tensor-memory accumulators in flight
constexpr uint32_t kScanTmemCols = 512;    // D buffer j: cols 160j .. 160j+159
constexpr float kTcErr = 1.6e-5f;          // 2^-16 + 2^-19 + fp64 rounding, rounded up

struct ScanSmem {
  uint8_t stage[kStages][kStageStride];    // keys, then query pieces; 1024-aligned
  uint8_t qp[kQpBytes];                    // the current sequence's pieces (query group)
  float uq[2][kMaxIdxHeads][128];          // [epilogue group]: |w'_h| (|q1_hc| + |r1_hc|)
  int64_t seq_items[kSeqCache];            // items of the first sequences (read once)
  int32_t n_seq_cached;
  float red[2][4];
  uint64_t full[kStages], empty[kStages], hdr[kStages];
  uint64_t d_full[kDBufs], d_empty[kDBufs];
  uint32_t tmem_slot;
  float qmax[3][kMaxIdxHeads];             // [group: query, epilogue 0, epilogue 1]: max |q_h|
  float qerr[2][kMaxIdxHeads];             // [epilogue group]: per-head sum of split errors
  float wq[2][kMaxIdxHeads];               // [epilogue group]: w_h 2^-e_h
  float unorm[2];                          // [epilogue group]: ||u||_2, rounded up
  float q_extra[2];
  volatile int32_t abort_flag;
};

__device__ inline uint32_t e4m3_rn(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return uint32_t(r) & 0xFF;
}

__device__ inline float e4m3_val(uint32_t code) {
  uint32_t h2 = e4m3x2_to_f16x2(uint16_t(code));
  return __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFF)));
}

__device__ inline int head_shift(float qm) { return qm > 0.0f ? max(-60, min(60, 7 - ilogbf(qm))) : 0; }

// Per-sequence query split, run by one 128-thread group (gt = 0..127; thread
// gt owns head gt/8, channels 16*(gt%8) .. +15; named barrier `bar_id`):
//   e_h: max |q_h| 2^e_h in [2^7, 2^8);  Qs = q 2^e_h = q1 + r1 (E4M3 pieces);
//   err_h = sum_c |Qs - q1 - r1| (nonzero only where r1 underflows E4M3).
// The query group (operands = true) writes q1 and r1 as 32 rows of the
// 128-byte swizzled K-major layout into sm.qp; the epilogue group (operands
// = false) derives w'_h = w_h 2^-e_h, ||u||_2 with u_c = sum_h |w'_h|
// (|q1_hc| + |r1_hc|), and the query rounding term 448 sum_h |w'_h| err_h,
// all rounded up where they bound an error.
__device__ void query_split(const IdxArgs& a, ScanSmem& sm, int b, int gt, int grp, int bar_id) {
  const int hi = a.d.idx_heads;
  const bool operands = grp == 0;
  const int eg = grp - 1;                                  // epilogue group
  const int h = gt >> 3, c0 = (gt & 7) * 16;
  // the query row piece and the weights are loaded before anything waits
  uint32_t wds[8] = {0, 0, 0, 0, 0, 0, 0, 0};          // bf16 pairs (the query is 4-byte aligned)
  if (h < hi) {
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint16_t*>(a.idx_q) +
                                                             (int64_t(b) * hi + h) * 128 + c0);
#pragma unroll
    for (int i = 0; i < 8; ++i) wds[i] = __ldg(qrow + i);
  }
  const float w_h = (!operands && h < hi) ? __ldg(a.w + int64_t(b) * hi + h) : 0.0f;
  const float w_g = (!operands && gt < hi) ? __ldg(a.w + int64_t(b) * hi + gt) : 0.0f;
  if (gt < kMaxIdxHeads) {
    sm.qmax[grp][gt] = 0.0f;
    if (!operands) sm.qerr[eg][gt] = 0.0f;
  }
  group_sync(bar_id);
  float qv[16];
  float mx = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    qv[i] = bf16_to_f32(uint16_t(wds[i >> 1] >> (16 * (i & 1))));
    mx = fmaxf(mx, fabsf(qv[i]));
  }
  atomicMax(reinterpret_cast<int*>(&sm.qmax[grp][h]), __float_as_int(mx));
  group_sync(bar_id);
  const int e = head_shift(sm.qmax[grp][h]);
  const float wabs = fabsf(ldexpf(w_h, -e));
  uint32_t w1[4] = {0, 0, 0, 0}, w2[4] = {0, 0, 0, 0};
  float err = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float x = ldexpf(qv[i], e);                     // exact: a power-of-two scaling
    const uint32_t c1 = e4m3_rn(x);
    const float d1 = e4m3_val(c1);
    const float r = x - d1;                                // exact
    const uint32_t c2 = e4m3_rn(r);
    const float d2 = e4m3_val(c2);
    err = __fadd_ru(err, fabsf(r - d2));                   // r - d2 exact
    if (!operands) sm.uq[eg][h][c0 + i] = __fmul_ru(wabs, fabsf(d1) + fabsf(d2));   // the sum is exact
    w1[i >> 2] |= c1 << (8 * (i & 3));
    w2[i >> 2] |= c2 << (8 * (i & 3));
  }
  if (operands) {
    const uint32_t chunk = uint32_t(c0 >> 4);
    *reinterpret_cast<uint4*>(sm.qp + tc::sw128_offset(h, chunk)) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
    *reinterpret_cast<uint4*>(sm.qp + tc::sw128_offset(16 + h, chunk)) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
    group_sync(bar_id);
    return;
  }
  if (err > 0.0f) atomicAdd(&sm.qerr[eg][h], err);
  if (gt < kMaxIdxHeads) sm.wq[eg][gt] = ldexpf(w_g, -head_shift(sm.qmax[grp][gt]));
  group_sync(bar_id);
  // ||u||^2: channel gt's u_c, squared and summed over the group, rounded up
  float uc = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxIdxHeads; ++i) uc = __fadd_ru(uc, sm.uq[eg][i][gt]);
  float sq = __fmul_ru(uc, uc);
#pragma unroll
  for (int o = 16; o; o >>= 1) sq = __fadd_ru(sq, __shfl_xor_sync(0xFFFFFFFFu, sq, o));
  if ((gt & 31) == 0) sm.red[eg][gt >> 5] = sq;
  group_sync(bar_id);
  if (gt == 0) {
    const float* rd = sm.red[eg];
    sm.unorm[eg] = __fsqrt_ru(__fadd_ru(__fadd_ru(rd[0], rd[1]), __fadd_ru(rd[2], rd[3])));
    float x = 0.0f;
    for (int i = 0; i < hi; ++i) x = __fmaf_ru(fabsf(sm.wq[eg][i]), __fmul_ru(sm.qerr[eg][i], 1.001f), x);
    sm.q_extra[eg] = __fmul_ru(x, 448.0f);
  }
  group_sync(bar_id);
}

// Whether row r of the tile is a position to score (issued before the
// epilogue waits for the MMA, so that its loads overlap the wait).
__device__ inline bool row_valid(const IdxArgs& a, bool reindex, const TileRef& pt, int r) {
  if (r >= pt.nvalid) return false;
  if (!reindex) return true;
  const bool paged = a.page_table != nullptr;
  const int64_t n_ctx = checked_ctx(a.ctx_len, a.d, pt.b, paged, a.ws);
  const int64_t item = pt.t0 + r;
  const int32_t blk = __ldg(a.pool_in + int64_t(pt.b) * a.d.pool_blocks + (item >> 3));
  const int64_t t = int64_t(blk) * kBlock + (item & 7);
  return blk >= 0 && t < n_ctx && kv_row(a.page_table, a.d, pt.b, int64_t(blk) * kBlock, a.ws) >= 0;
}

// Both 32-column loads of a row, then one wait.
__device__ inline void tmem_ld32x2(uint32_t ta, uint32_t tb, float (&va)[32], float (&vb)[32]) {
  uint32_t ra[32], rb[32];
#define CSA2_LD32(R, T)                                                                                 \
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "                                               \
               "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "                \
               "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];" \
               : "=r"(R[0]), "=r"(R[1]), "=r"(R[2]), "=r"(R[3]), "=r"(R[4]), "=r"(R[5]), "=r"(R[6]),      \
                 "=r"(R[7]), "=r"(R[8]), "=r"(R[9]), "=r"(R[10]), "=r"(R[11]), "=r"(R[12]), "=r"(R[13]),  \
                 "=r"(R[14]), "=r"(R[15]), "=r"(R[16]), "=r"(R[17]), "=r"(R[18]), "=r"(R[19]),            \
                 "=r"(R[20]), "=r"(R[21]), "=r"(R[22]), "=r"(R[23]), "=r"(R[24]), "=r"(R[25]),            \
                 "=r"(R[26]), "=r"(R[27]), "=r"(R[28]), "=r"(R[29]), "=r"(R[30]), "=r"(R[31])             \
               : "r"(T))
  CSA2_LD32(ra, ta);
  CSA2_LD32(rb, tb);
#undef CSA2_LD32
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) { va[i] = __uint_as_float(ra[i]); vb[i] = __uint_as_float(rb[i]); }
}

// Epilogue of one tile for the thread owning row r (TMEM lanes of warp
// quarter q = r / 32) of epilogue group eg: scores, bounds, block maxima,
// writes.
__device__ inline void scan_epilogue(const IdxArgs& a, bool reindex, const ScanSmem& sm, int eg,
                                     const TileRef& pt, uint32_t tmem_d, bool valid, int r, int lane) {
  float dv[32], gv[32];
  tmem_ld32x2(tmem_d + kTile, tmem_d + (r & ~31), dv, gv);   // k . q1_h, k . r1_h; Gram columns
  float g = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) g = i == lane ? gv[i] : g;   // the diagonal element
  float v = 0.0f;
#pragma unroll
  for (int h = 0; h < 16; ++h) v = __fmaf_rn(sm.wq[eg][h], fmaxf(dv[h] + dv[16 + h], 0.0f), v);
  // ||k||^2 from the MMA is low by at most 2^-14 of itself: raise it by 2^-13
  const float knorm = __fsqrt_ru(__fmul_ru(fmaxf(g, 0.0f), 1.0f + 0x1p-13f));
  float delta = __fadd_ru(__fmul_ru(__fmul_ru(__fmul_ru(knorm, sm.unorm[eg]), 1.0003f), kTcErr), sm.q_extra[eg]);
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
  if ((lane & 7) == 0 && valid) {
    int64_t j = t >> 3;
    ws_f[(a.L.blk_scores >> 2) + int64_t(pt.b) * a.L.nb_max + j] = bmax;
    ws_f[(a.L.blk_delta >> 2) + int64_t(pt.b) * a.L.nb_max + j] = bd;
  }
}

__global__ void __launch_bounds__(kScanThreads, 1)
    scan_tc_kernel(IdxArgs a, const __grid_constant__ CUtensorMap kmap, bool reindex) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  ScanSmem& sm = *reinterpret_cast<ScanSmem*>(
      smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  __shared__ int64_t total_tiles_s;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // early inputs: the lengths and the keys may be read before the previous
  // kernel finishes; everything else waits for it (below)
  if (!a.early) {
    pdl_wait();
    pdl_launch_dependents();
  }
  // ---- tiles of all sequences, this CTA's contiguous share ----------------------
  if (wid == 0) {
    const int64_t tsum = count_tiles(a, sm, reindex, lane);
    if (lane == 0) total_tiles_s = tsum;
  }
  __syncthreads();
  const int64_t T = total_tiles_s;
  const int64_t g0 = int64_t(blockIdx.x) * T / gridDim.x;
  const int64_t g1 = int64_t(blockIdx.x + 1) * T / gridDim.x;
  if (g0 >= g1) return;

  if (wid == 0) tc::tmem_alloc(&sm.tmem_slot, kScanTmemCols);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&sm.full[s], 1);                    // the producer's arrival (with its TMA bytes)
      tc::mbar_init(&sm.empty[s], 1);
      tc::mbar_init(&sm.hdr[s], 4);
    }
    for (int i = 0; i < kDBufs; ++i) {
      tc::mbar_init(&sm.d_full[i], 1);
      tc::mbar_init(&sm.d_empty[i], 4);
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
    // the producer (warp 0) waits once its first ring of keys is in flight
    pdl_wait();
    pdl_launch_dependents();
  }

  if (wid == 0 && reindex) {
    // ================= producer: TMA gather of pool blocks =================
    produce_reindex<128, kStages>(a, &kmap, sm, sm.stage[0], kStageStride, sm.full, sm.empty, g0, ntiles, lane,
                                  a.early != 0);
  } else if (wid == 0) {
    // ================= producer: TMA ring =================
    if (lane == 0)
      produce_full<128, kStages>(a, &kmap, sm, sm.stage[0], kStageStride, sm.full, sm.empty, g0, ntiles, a.early != 0);
  } else if (wid == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3(kTile, kMmaN);
      // descriptors are formed once; an offset of x bytes adds x/16 to the
      // start-address field (every operand lies below 256 KB, so it never carries)
      const uint64_t d0 = tc::smem_desc(tc::smem_u32(sm.stage[0]), 16, 1024, 2);
      int issued = 0;
      RingPos<kStages> ring;
      for (int k = 0; k < ntiles; ++k, ring.next()) {
        const int stage = ring.stage;
        const int buf = k % kDBufs;
        if (!wait_or_abort(sm, &sm.full[stage], ring.phase)) break;   // keys
        if (!wait_or_abort(sm, &sm.hdr[stage], ring.phase)) break;    // query pieces
        if (k >= kDBufs && !wait_or_abort(sm, &sm.d_empty[buf], uint32_t((k / kDBufs - 1) & 1))) break;
        tc::tc_fence_after_sync();
        const uint64_t ds = d0 + uint64_t(stage) * (kStageStride >> 4);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)                   // K = 32 E4M3 (32 bytes) per step
          mma_f8(tmem + kMmaN * buf, ds + 2 * ks, ds + 2 * ks, idesc, ks > 0);
        tc::mma_commit(&sm.empty[stage]);
        tc::mma_commit(&sm.d_full[buf]);
        issued = k + 1;
      }
      // after an abort, let the issued MMAs finish before the tensor memory is freed
      if (sm.abort_flag && issued > 0)
        tc::mbar_wait_bounded(&sm.d_full[(issued - 1) % kDBufs], uint32_t(((issued - 1) / kDBufs) & 1),
                              20ull * 1000 * 1000);
    }
  } else if (wid < 6) {
    // ================= query group (warps 2-5): pieces behind each tile's keys =====
    const int gt = tid - 64;
    int cb = 0, cur_b = -1;
    int64_t cbase = 0;
    RingPos<kStages> ring;
    for (int k = 0; k < ntiles; ++k, ring.next()) {
      const TileRef tr = tile_of(a, sm, reindex, g0 + k, cb, cbase);
      const int stage = ring.stage;
      if (tr.b != cur_b) {
        query_split(a, sm, tr.b, gt, 0, 1);
        cur_b = tr.b;
      }
      // the stage is free once the MMAs of its previous tile completed
      if (k >= kStages && !wait_or_abort(sm, &sm.empty[stage], ring.phase ^ 1u)) break;
      const uint4* src = reinterpret_cast<const uint4*>(sm.qp);
      uint4* dst = reinterpret_cast<uint4*>(sm.stage[stage] + kKeyBytes);
#pragma unroll
      for (int i = 0; i < kQpBytes / 16 / kGroupThreads; ++i) dst[gt + i * kGroupThreads] = src[gt + i * kGroupThreads];
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) arrive(&sm.hdr[stage]);
    }
  } else {
    // ================= epilogue groups (warps 6-9: even tiles, 10-13: odd) ==========
    const int eg = (wid - 6) >> 2;
    const int gt = tid - 192 - eg * kGroupThreads;
    const int quarter = wid & 3;                      // TMEM lanes 32*quarter ..
    const int r = quarter * 32 + lane;                // row of the tile
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    int cb = 0, cur_b = -1;
    int64_t cbase = 0;
    for (int k = eg; k < ntiles; k += 2) {
      const TileRef tr = tile_of(a, sm, reindex, g0 + k, cb, cbase);
      if (tr.b != cur_b) {
        query_split(a, sm, tr.b, gt, 1 + eg, 2 + eg);
        cur_b = tr.b;
      }
      const bool valid = row_valid(a, reindex, tr, r);
      const int buf = k % kDBufs;
      if (!wait_or_abort(sm, &sm.d_full[buf], uint32_t((k / kDBufs) & 1))) break;
      tc::tc_fence_after_sync();
      scan_epilogue(a, reindex, sm, eg, tr, tmem + lane_base + kMmaN * buf, valid, r, lane);
      tc::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) arrive(&sm.d_empty[buf]);
    }
  }
  tc::tc_fence_before_sync();
  __syncthreads();
  if (sm.abort_flag && tid == 0) raise_err(a.ws, CSA2_DEV_TIMEOUT);
  if (wid == 0) tc::tmem_dealloc(tmem, kScanTmemCols);
}

// ---------------------------------------------------------------------------
// Host side: tensor map over the indexer-K cache and the launch
// ---------------------------------------------------------------------------
cudaError_t launch_scan_tc(const IdxArgs& a, bool reindex, cudaStream_t st) {
  CUtensorMap map;
  cudaError_t e = idx_key_map(&map, a, reindex, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  const int64_t grid = scan_grid(a, reindex);
  const size_t smem = sizeof(ScanSmem) + 1024;
  static KernelAttrs done;
  e = prepare_kernel(scan_tc_kernel, smem, false, done);
  if (e != cudaSuccess) return e;
  CSA2_PROFILED(st, reindex ? "reindex_score_tc" : "indexer_scan_tc",
                (e = launch_pdl(scan_tc_kernel, dim3(unsigned(grid)), dim3(kScanThreads), smem, st, 1, a, map,
                                reindex)));
  return e;
}

}  // namespace csa2
