// scan.cu -- Full-mode indexer scan on the tcgen05 tensor cores (E4M3 keys).
//
// For every visible position t (foosynaptic atlas "DeepSeek-V4.1-Flash 梗概",
// section 3.2: the first Full layer scores every causally visible position):
//   d_{t,h} = q_h . k_t,  s_t = sum_h w_h ReLU(d_{t,h}),  bs_j = max over block j,
// and a rigorous bound delta_j >= |s_t - v_t| for the approximate v_t.
//
// Work: persistent CTAs walk contiguous ranges of 128-position tiles.
//   * TMA (tensor map, 128-byte swizzle) streams each tile's 128 x 128 B of
//     E4M3 keys into a 4-stage shared-memory ring.
//   * 8 warps convert the keys to f16 (exact: E4M3 is a subset of f16) and
//     store them into tensor memory as the MMA's A operand, together with
//     their absolute values |A|.
//   * One thread issues D = A . Qf^T and D2 = |A| . |Qf|^T (M=128 positions,
//     N=16 heads, K=128, f16 in, fp32 accumulation).  Qf = q_h * 2^e_h in f16,
//     with a per-head power of two e_h so that every bf16 query element lands
//     in f16's exact range (the rare element that does not is counted in the
//     bound).
//   * The epilogue reads D and D2 from tensor memory: v_t = sum_h w'_h
//     ReLU(D_h) with w'_h = w_h 2^-e_h, and delta_t = C * sum_h |w'_h| D2_h
//     + (query rounding term), C covering the tensor-core accumulation error
//     (modelled as at most 2^-14 of sum|products| per head dot), the fp32
//     head sum and the fp64 rounding of the exact score.  Block max of v and
//     delta over 8 positions are written with the position scores.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"
#include "profile.cuh"
#include "tc.cuh"

namespace csa2 {

constexpr int kScanThreads = 256;
constexpr int kTile = 128;                 // positions per tile (= MMA M)
constexpr int kStages = 4;                 // TMA ring depth
constexpr int kStageBytes = kTile * 128;   // 16 KB of E4M3 keys
constexpr uint32_t kScanTmemCols = 256;
// tensor-memory columns
constexpr uint32_t kColA = 0, kColAbs = 64, kColD = 128;   // D[buf] at 128 + 32 buf, D2 at +16

// Error-model constant of the tensor-core scores (see file comment).
constexpr float kTcErr = 6.3e-5f;          // 2^-14 + 2^-19 + fp64 rounding, rounded up

struct ScanSmem {
  uint8_t stage[kStages][kStageBytes];     // 1024-aligned (swizzle atoms)
  uint8_t qf[2][16 * 128];                 // f16 query [16 heads][128], 2 regions of 64 ch
  uint8_t qa[2][16 * 128];                 // |query|, same layout
  uint64_t full[kStages];
  uint64_t dbar[2];
  uint32_t tmem_slot;
  int32_t cur_b;
  float wq[kMaxIdxHeads];                  // w_h * 2^-e_h
  float wq_abs[kMaxIdxHeads];
  float qmax_bits[kMaxIdxHeads];
  float qerr[kMaxIdxHeads];
  float q_extra;
  int32_t abort_flag;
};

__device__ inline void tma_load_box(const CUtensorMap* map, uint8_t* dst, int32_t row, uint64_t* bar) {
  tc::tma_load_2d(map, dst, 0, row, bar);
}

__device__ inline void mbar_expect_tx(uint64_t* bar, uint32_t bytes) { tc::mbar_expect_tx(bar, bytes); }

__device__ inline void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
      ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
        "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// D (+)= A[tmem] . B[smem]^T
__device__ inline void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                  bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(uint32_t(accumulate))
      : "memory");
}

// f16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

struct TileRef {
  int b;
  int64_t t0;        // first position
  int nvalid;        // valid positions in the tile
};

// Global tile g -> (sequence, first position); tiles of sequence b are
// ceil(N_b / 128).  Linear walk from a hint (tiles are visited in order).
// Items of sequence b: its positions (Full) or its pool positions, 8 per pool
// block (Reindex).
__device__ inline int64_t scan_items(const IdxArgs& a, int b, bool reindex) {
  if (reindex) {
    int64_t plen = __ldg(a.pool_len_in + b);
    return (plen < 0 || plen > a.d.pool_blocks) ? 0 : plen * kBlock;
  }
  int64_t n = __ldg(a.ctx_len + b);
  const bool paged = a.page_table != nullptr;
  if (n < 0 || n > a.d.max_ctx || (paged && n > int64_t(a.d.max_pages) * kPage)) n = 0;
  return n;
}

__device__ inline TileRef tile_of(const IdxArgs& a, bool reindex, int64_t g, int& hint_b,
                                  int64_t& hint_base) {
  while (true) {
    int64_t n = scan_items(a, hint_b, reindex);
    int64_t nt = (n + kTile - 1) / kTile;
    if (g < hint_base + nt) {
      TileRef r;
      r.b = hint_b;
      r.t0 = (g - hint_base) * kTile;
      r.nvalid = int(min64(kTile, n - r.t0));
      return r;
    }
    hint_base += nt;
    ++hint_b;
  }
}

__device__ inline void issue_tile_load(const IdxArgs& a, bool reindex, const CUtensorMap* map,
                                       ScanSmem& sm, const TileRef& tr, int stage) {
  if (reindex) {
    // one 8-row box per pool block (a block never crosses a 64-position page)
    const bool paged = a.page_table != nullptr;
    const int64_t n_ctx = checked_ctx(a.ctx_len, a.d, tr.b, paged, a.ws);
    const int nblk = (tr.nvalid + kBlock - 1) / kBlock;
    int32_t rows[kTile / kBlock];
    uint32_t bytes = 0;
    for (int j = 0; j < nblk; ++j) {
      int32_t blk = __ldg(a.pool_in + int64_t(tr.b) * a.d.pool_blocks + (tr.t0 >> 3) + j);
      int64_t row = -1;
      if (blk >= 0 && int64_t(blk) * kBlock < n_ctx) row = kv_row(a.page_table, a.d, tr.b, int64_t(blk) * kBlock, a.ws);
      rows[j] = int32_t(row);
      if (row >= 0) bytes += kBlock * 128;
    }
    mbar_expect_tx(&sm.full[stage], bytes);
    for (int j = 0; j < nblk; ++j)
      if (rows[j] >= 0) tma_load_box(map, sm.stage[stage] + j * kBlock * 128, rows[j], &sm.full[stage]);
    return;
  }
  uint32_t bytes = 0;
  int32_t rows[2];
  int nbox = (tr.nvalid > 64) ? 2 : 1;
  for (int h = 0; h < nbox; ++h) {
    int64_t t = tr.t0 + 64 * h;
    int64_t row = kv_row(a.page_table, a.d, tr.b, t, a.ws);
    rows[h] = int32_t(row);
    if (row >= 0) bytes += 64 * 128;
  }
  mbar_expect_tx(&sm.full[stage], bytes);
  for (int h = 0; h < nbox; ++h)
    if (rows[h] >= 0) tma_load_box(map, sm.stage[stage] + h * 64 * 128, rows[h], &sm.full[stage]);
}

// Per-sequence query operands: Qf = q * 2^e_h (f16) and |Qf|, 128-byte
// swizzled K-major (16 rows, 2 regions of 64 channels); the weights
// w'_h = w_h 2^-e_h; and the query-rounding term of the bound.
__device__ void build_query(const IdxArgs& a, ScanSmem& sm, int b) {
  const int tid = threadIdx.x, hi = a.d.idx_heads;
  if (tid < kMaxIdxHeads) { sm.qmax_bits[tid] = 0.0f; sm.qerr[tid] = 0.0f; }
  __syncthreads();
  const int h = tid >> 4, c0 = (tid & 15) * 8;            // 16 heads x 16 chunks of 8 channels
  float qv[8];
  float mx = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    qv[i] = h < hi ? bf16_to_f32(reinterpret_cast<const uint16_t*>(a.idx_q)[(int64_t(b) * hi + h) * 128 + c0 + i]) : 0.0f;
    mx = fmaxf(mx, fabsf(qv[i]));
  }
  atomicMax(reinterpret_cast<int*>(&sm.qmax_bits[h]), __float_as_int(mx));
  __syncthreads();
  float qm = sm.qmax_bits[h];
  int e = 0;
  if (qm > 0.0f) e = 14 - ilogbf(qm);                      // max |q| * 2^e in [2^14, 2^15)
  uint32_t wf[4], wa[4];
  float err = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float x0 = ldexpf(qv[2 * i], e), x1 = ldexpf(qv[2 * i + 1], e);
    __half2 hv = __floats2half2_rn(x0, x1);
    err = __fadd_ru(err, fabsf(__low2float(hv) - x0));
    err = __fadd_ru(err, fabsf(__high2float(hv) - x1));
    wf[i] = *reinterpret_cast<uint32_t*>(&hv);
    wa[i] = wf[i] & 0x7FFF7FFFu;
  }
  const uint32_t region = c0 >> 6, chunk = (c0 & 63) >> 3;
  const uint32_t off = tc::sw128_offset(h, chunk);
  *reinterpret_cast<uint4*>(sm.qf[region] + off) = make_uint4(wf[0], wf[1], wf[2], wf[3]);
  *reinterpret_cast<uint4*>(sm.qa[region] + off) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
  if (err > 0.0f) atomicAdd(&sm.qerr[h], err);
  __syncthreads();
  if (tid < kMaxIdxHeads) {
    float w = tid < hi ? a.w[int64_t(b) * hi + tid] : 0.0f;
    float qm2 = sm.qmax_bits[tid];
    int e2 = qm2 > 0.0f ? 14 - ilogbf(qm2) : 0;
    sm.wq[tid] = ldexpf(w, -e2);
    sm.wq_abs[tid] = fabsf(sm.wq[tid]);
  }
  __syncthreads();
  if (tid == 0) {
    // |Qf - q 2^e| summed per head, times the largest E4M3 magnitude
    float x = 0.0f;
    for (int i = 0; i < hi; ++i) x = __fmaf_ru(sm.wq_abs[i], __fmul_ru(sm.qerr[i], 1.001f), x);
    sm.q_extra = __fmul_ru(x, 448.0f);
    sm.cur_b = b;
  }
  tc::fence_proxy_async_smem();
  __syncthreads();
}

// Epilogue of one tile for the thread owning row r (warps of half 0): scores,
// bounds, block maxima, writes.
__device__ inline void scan_epilogue(const IdxArgs& a, bool reindex, const ScanSmem& sm,
                                     const TileRef& pt, uint32_t tmem_d, int r, int lane) {
  float dv[16], d2[16];
  tc::tmem_ld16(tmem_d, dv);
  tc::tmem_ld16(tmem_d + 16, d2);
  bool valid = r < pt.nvalid;
  if (reindex && valid) {
    const bool paged = a.page_table != nullptr;
    const int64_t n_ctx = checked_ctx(a.ctx_len, a.d, pt.b, paged, a.ws);
    const int64_t item = pt.t0 + r;
    int32_t blk = __ldg(a.pool_in + int64_t(pt.b) * a.d.pool_blocks + (item >> 3));
    int64_t t = int64_t(blk) * kBlock + (item & 7);
    valid = blk >= 0 && t < n_ctx && kv_row(a.page_table, a.d, pt.b, int64_t(blk) * kBlock, a.ws) >= 0;
  }
  float v = 0.0f, bnd = 0.0f;
#pragma unroll
  for (int h = 0; h < 16; ++h) {
    v = __fmaf_rn(sm.wq[h], fmaxf(dv[h], 0.0f), v);
    bnd = __fmaf_ru(sm.wq_abs[h], d2[h], bnd);
  }
  float delta = __fadd_ru(__fmul_ru(__fmul_ru(bnd, 1.0003f), kTcErr), sm.q_extra);
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

__global__ void __launch_bounds__(kScanThreads, 2)
    scan_tc_kernel(IdxArgs a, const __grid_constant__ CUtensorMap kmap, bool reindex) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  ScanSmem& sm = *reinterpret_cast<ScanSmem*>(
      smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  __shared__ int64_t total_tiles_s;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int quarter = wid & 3, half = wid >> 2;
  // ---- tiles of all sequences, this CTA's contiguous share ----------------------
  if (wid == 0) {
    int64_t tsum = 0;
    for (int b = lane; b < a.batch; b += 32) tsum += (scan_items(a, b, reindex) + kTile - 1) / kTile;
#pragma unroll
    for (int o = 16; o; o >>= 1) tsum += __shfl_xor_sync(0xFFFFFFFFu, tsum, o);
    if (lane == 0) total_tiles_s = tsum;
  }
  __syncthreads();
  const int64_t T = total_tiles_s;
  const int64_t g0 = int64_t(blockIdx.x) * T / gridDim.x;
  const int64_t g1 = int64_t(blockIdx.x + 1) * T / gridDim.x;
  if (g0 >= g1) return;

  if (wid == 0) tc::tmem_alloc(&sm.tmem_slot, kScanTmemCols);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) tc::mbar_init(&sm.full[s], 1);
    tc::mbar_init(&sm.dbar[0], 1);
    tc::mbar_init(&sm.dbar[1], 1);
    tc::fence_mbar_init();
    sm.cur_b = -1;
    sm.abort_flag = 0;
  }
  tc::tc_fence_before_sync();
  __syncthreads();
  tc::tc_fence_after_sync();
  const uint32_t tmem = sm.tmem_slot;
  constexpr uint32_t idesc = idesc_f16(kTile, 16);
  const int r = quarter * 32 + lane;                 // this thread's row of the tile
  const uint32_t lane_base = uint32_t(quarter * 32) << 16;

  // producer (thread 0): the first kStages tiles
  int pb = 0;
  int64_t pbase = 0, next_load = g0;
  if (tid == 0) {
    for (int s = 0; s < kStages && next_load < g1; ++s, ++next_load)
      issue_tile_load(a, reindex, &kmap, sm, tile_of(a, reindex, next_load, pb, pbase), s);
  }
  int cb = 0;
  int64_t cbase = 0;
  TileRef prev = {0, 0, 0};
  bool pending = false;
  int64_t k = 0;
  for (int64_t g = g0; g < g1; ++g, ++k) {
    const TileRef tr = tile_of(a, reindex, g, cb, cbase);
    const int stage = int(k % kStages);
    const uint32_t buf = uint32_t(k & 1);
    // ---- this thread's 64 channels of its row, E4M3 -> f16 (exact) ----------
    if (!tc::mbar_wait_bounded(&sm.full[stage], uint32_t((k / kStages) & 1))) sm.abort_flag = 1;
    uint32_t af[32], aa[32];
    const uint8_t* srow = sm.stage[stage] + r * 128;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t c = half * 4 + j;
      uint4 v = *reinterpret_cast<const uint4*>(srow + ((c ^ (uint32_t(r) & 7u)) << 4));
      uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          uint32_t f = e4m3x2_to_f16x2(uint16_t(w4[i] >> (16 * p)));
          af[j * 8 + i * 2 + p] = f;
          aa[j * 8 + i * 2 + p] = f & 0x7FFF7FFFu;
        }
      }
    }
    // ---- the previous tile's MMAs read A: wait for them ---------------------
    if (pending) {
      if (!tc::mbar_wait_bounded(&sm.dbar[buf ^ 1u], uint32_t(((k - 1) >> 1) & 1))) sm.abort_flag = 1;
      tc::tc_fence_after_sync();
    }
    if (tr.b != sm.cur_b) {
      // new sequence: finish the previous tile with its own weights, then
      // build this sequence's query operands
      if (pending && half == 0) scan_epilogue(a, reindex, sm, prev, tmem + lane_base + kColD + 32 * (buf ^ 1u), r, lane);
      pending = false;
      tc::tc_fence_before_sync();
      __syncthreads();
      build_query(a, sm, tr.b);
    }
    tmem_st32(tmem + lane_base + kColA + half * 32, af);
    tmem_st32(tmem + lane_base + kColAbs + half * 32, aa);
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    tc::tc_fence_before_sync();
    __syncthreads();
    const bool abort_now = sm.abort_flag != 0;
    // ---- this tile's MMAs (one thread); refill the consumed stage ----------------
    if (tid == 0 && !abort_now) {
      tc::tc_fence_after_sync();
      const uint32_t qf0 = tc::smem_u32(sm.qf[0]), qa0 = tc::smem_u32(sm.qa[0]);
      const uint32_t dcol = tmem + kColD + 32 * buf;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t boff = (ks >> 2) * (16 * 128) + (ks & 3) * 32;
        mma_f16_ts(dcol, tmem + kColA + 8 * ks, tc::smem_desc(qf0 + boff, 16, 1024, 2), idesc, ks > 0);
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t boff = (ks >> 2) * (16 * 128) + (ks & 3) * 32;
        mma_f16_ts(dcol + 16, tmem + kColAbs + 8 * ks, tc::smem_desc(qa0 + boff, 16, 1024, 2), idesc, ks > 0);
      }
      tc::mma_commit(&sm.dbar[buf]);
      if (next_load < g1) {
        issue_tile_load(a, reindex, &kmap, sm, tile_of(a, reindex, next_load, pb, pbase), stage);
        ++next_load;
      }
    }
    if (abort_now) break;
    if (pending && half == 0) scan_epilogue(a, reindex, sm, prev, tmem + lane_base + kColD + 32 * (buf ^ 1u), r, lane);
    prev = tr;
    pending = true;
  }
  // ---- the last tile ------------------------------------------------------------------
  if (pending && !sm.abort_flag) {
    const uint32_t buf = uint32_t((k - 1) & 1);
    bool ok = tc::mbar_wait_bounded(&sm.dbar[buf], uint32_t(((k - 1) >> 1) & 1));
    tc::tc_fence_after_sync();
    if (ok && half == 0) scan_epilogue(a, reindex, sm, prev, tmem + lane_base + kColD + 32 * buf, r, lane);
    if (!ok) sm.abort_flag = 1;
  }
  tc::tc_fence_before_sync();
  __syncthreads();
  if (sm.abort_flag && tid == 0) raise_err(a.ws, CSA2_DEV_TIMEOUT);
  if (wid == 0) tc::tmem_dealloc(tmem, kScanTmemCols);
}

// ---------------------------------------------------------------------------
// Host side: tensor map over the indexer-K cache and the launch
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

cudaError_t launch_scan_tc(const IdxArgs& a, bool reindex, cudaStream_t st) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const bool paged = a.page_table != nullptr;
  const uint64_t rows = paged ? uint64_t(a.d.num_pages) * kPage : uint64_t(a.batch) * uint64_t(a.d.max_ctx);
  CUtensorMap map;
  cuuint64_t gdim[2] = {128, rows};
  cuuint64_t gstride[1] = {128};
  cuuint32_t box[2] = {128, reindex ? uint32_t(kBlock) : 64u};   // one pool block / half a tile
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a.idx_k), gdim, gstride, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // the tile count is known only on the device; the grid is sized for an
  // upper bound and the CTAs split the actual tiles evenly
  int64_t items_ub = reindex ? int64_t(a.d.pool_blocks) * kBlock : a.d.max_ctx;
  int64_t tiles_ub = int64_t(a.batch) * ((items_ub + kTile - 1) / kTile);
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  size_t smem = sizeof(ScanSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  int64_t grid = min64(int64_t(2) * sms, tiles_ub);
  if (grid < 1) grid = 1;
  CSA2_PROFILED(st, reindex ? "reindex_score_tc" : "indexer_scan_tc",
                (scan_tc_kernel<<<unsigned(grid), kScanThreads, smem, st>>>(a, map, reindex)));
  return cudaGetLastError();
}

}  // namespace csa2
