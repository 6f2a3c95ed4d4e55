// select.cu -- certified Top-P / Top-K selection of the CSA2 indexer.
//
// Picks the P best items (blocks for the candidate pool, positions for the
// Top-K) under the order (exact score desc, index asc), given approximate
// scores v with a rigorous bound |v - s| <= delta (foosynaptic atlas
// "DeepSeek-V4.1-Flash 梗概", section 3.2: the Full layer keeps the Top-2048
// blocks of 8 as the pool, Reindex layers take Top-512 inside it).
//
//   U = v + delta (rounded up), L = v - delta (rounded down)
//   A radix select on v alone finds a bucket [v_lo, v_hi] holding the P-th
//   largest v; with D = max delta over the items, the P-th largest U is at
//   most v_hi + D and the P-th largest L at least v_lo - D, so
//   mu'     = v_hi + D (rounded up)   >= P-th largest U
//   lambda' = v_lo - D (rounded down) <= P-th largest L
//   L > mu'              -> selected (its exact score beats the P-th best)
//   U < lambda'          -> not selected
//   otherwise ("band")   -> exact score (fixed point, exact.cuh), then the
//                           best (P - #selected) band items by exact score.
// The result is the selection on exact scores.
//
// One CTA holds up to 16,384 items in shared memory; a sequence with more
// items (the block scores of a context above 131,072 positions) is split over
// a thread-block cluster of up to 8 CTAs that merge their radix histograms
// through distributed shared memory.  Cluster barriers are hardware barriers
// (no software spin).
//
// Full mode runs two selection sides at once (grid z) while both fit one
// wave of one CTA per SM.  Side 0 selects the pool.  Side 1 selects the
// Top-K positions from the blocks whose bounds let them be among the K best
// blocks (the certain ones and the band of a block selection with k = K,
// without exact re-scoring): a Top-K position's block is among the K best
// blocks, and these are in the pool when K <= P or the pool is every block.
// Otherwise (or for a larger batch) side 0 selects the pool and then the
// Top-K of its positions.  The positions of at most P blocks are selected by
// one CTA (rank 0 of a cluster).
#include <cooperative_groups.h>

#include "common.cuh"
#include "exact.cuh"
#include "fp4.cuh"
#include "kernels.cuh"
#include "profile.cuh"

namespace cg = cooperative_groups;

namespace csa2 {

enum ItemKind { kBlocks = 0, kPoolPos = 1, kReindexPos = 2 };

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
static_assert(kMaxPool % kSelThreads == 0, "pool ids per selection thread");
constexpr int kSortCap = 4096;
constexpr int kBins = 2048;                 // 11-bit radix digits
constexpr int kMaxSelCluster = 8;           // CTAs of a selection cluster
static_assert(kMaxCtx / kBlock <= int64_t(kMaxSelCluster) * kSelCapPerCta, "block items fit the cluster");
constexpr int kExItems = 128;               // band items re-scored per chunk (<= 8 positions each)
constexpr int kQiStride = 132;              // words per head row of the integer query (16-byte
                                            // loads of 16 heads spread over all banks)

struct SelSmem {
  uint32_t keyU[kSelCapPerCta];             // reused: sort keys (rank 0)
  uint32_t keyL[kSelCapPerCta];             // reused: band list, sort ids
  uint32_t band_bits[kSelCapPerCta / 32];
  uint32_t sel_bits[kSelCapPerCta / 32];
  uint32_t word_off[kSelCapPerCta / 32];
  uint32_t hist[2][kBins];                  // this CTA's histograms (U, L)
  uint32_t ghist[2][kBins];                 // cluster-wide sums
  Factor qf[kMaxIdxHeads * 128];            // query factors, [channel][head]
  __align__(16) int32_t qi[kMaxIdxHeads * kQiStride];   // query as integers, [head][channel]
  int32_t k_lut[256];                       // E4M3 byte -> its value * 2^9 (an exact integer)
  int32_t q_elo[kMaxIdxHeads];              // q = qi * 2^q_elo (exact)
  int32_t q_fast[kMaxIdxHeads];             // 1: the int32 x int32 -> int64 path is exact
  unsigned long long q_l1[kMaxIdxHeads];    // sum_c |qi|
  float w[kMaxIdxHeads];
  int32_t pool_ids[kMaxPool];
  uint32_t red[2][kSelWarps];
  uint32_t bucket, bucket_cnt, rem;
  uint32_t kmin, kmax, base_key;
  float dmax, dmax_all, dred[kSelWarps];
  uint32_t kmax_all;
  int shift0;
  uint32_t cnt_in, cnt_band, cnt_sel;
  uint32_t tot3[3];                         // cluster sums read once by warp 0
  uint32_t n_cand;
  int32_t fast_exact;                       // E4M3 keys, every head on the int64 path
};

// Scratch of the exact re-scoring, overlaid on keyU (free between the
// classification and the final pick).
constexpr int kExRows = 48;                // positions per round of the exact re-scoring
constexpr int kExRowWords = 132;          // 128 words + 4: 16-byte aligned rows
constexpr int kExSumThreads = 64;         // threads that form the ordered head sums
constexpr int kStageWords = 2;            // row words a staging thread loads per batch

constexpr int kFastRows = 64;             // positions of one pass of the E4M3 / FP4 re-scoring
constexpr int kExTailWords = 832;         // extends the work area for the E4M3 pass

struct ExScratch {
  double cand_score[kSelThreads];
  int64_t cand_pos[kSelThreads];            // candidate positions of a chunk
  unsigned long long item_best[128];
  int32_t cand_item[kSelThreads];
  // work area of the re-scoring (dd, krows and tail are contiguous; the E4M3
  // pass lays its own [kFastRows][kMaxIdxHeads] doubles and
  // [kFastRows][128] staged integers over all three)
  double dd[2][kExRows * kMaxIdxHeads];     // w_h * ReLU(d_h) of a round, double-buffered
  __align__(16) int32_t krows[kExRows * kExRowWords];   // staged keys: E4M3 as k*2^9 integers, or fp32 bits
  int32_t tail[kExTailWords];
};
static_assert(sizeof(ExScratch) <= sizeof(uint32_t) * kSelCapPerCta, "exact scratch must fit keyU");
static_assert(offsetof(ExScratch, krows) == offsetof(ExScratch, dd) + sizeof(ExScratch::dd) &&
              offsetof(ExScratch, tail) == offsetof(ExScratch, krows) + sizeof(ExScratch::krows),
              "contiguous work area");
static_assert(offsetof(ExScratch, dd) % 16 == 0, "16-byte aligned work area");
static_assert(sizeof(double) * kFastRows * kMaxIdxHeads + sizeof(int32_t) * kFastRows * 128 <=
              sizeof(ExScratch::dd) + sizeof(ExScratch::krows) + sizeof(ExScratch::tail), "E4M3 pass fits");

__device__ inline ExScratch& ex_scratch(SelSmem& sm) { return *reinterpret_cast<ExScratch*>(sm.keyU); }

struct SelCtx {
  int rank, cs;
  int64_t n_ctx;
  int b;
  int side;                                 // selection side: its band scratch in the workspace
};

__device__ inline void cl_sync(const SelCtx& c) {
  if (c.cs > 1) cg::this_cluster().sync(); else __syncthreads();
}

template <class T>
__device__ inline const T* remote(const SelCtx& c, const T* p, int r) {
  return c.cs > 1 ? cg::this_cluster().map_shared_rank(p, r) : p;
}

// Block-wide exclusive scan of word popcounts of `bits` (nwords <= 512) into
// sm.word_off; returns the total.
__device__ uint32_t scan_words(SelSmem& sm, const uint32_t* bits, int nwords) {
  __syncthreads();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  uint32_t v = tid < nwords ? __popc(bits[tid]) : 0;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm.red[0][wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t s = sm.red[0][lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += y;
    }
    sm.red[0][lane] = s;
  }
  __syncthreads();
  uint32_t base = wid ? sm.red[0][wid - 1] : 0;
  if (tid < nwords) sm.word_off[tid] = base + x - v;
  uint32_t total = sm.red[0][kSelWarps - 1];
  __syncthreads();
  return total;
}

// The bin (scanning from the top) of histogram h that holds the sm.rem-th
// largest key; sets sm.bucket and sm.bucket_cnt (its count) and updates
// sm.rem.  Thread t owns bins 2047-2t and 2046-2t.
static_assert(kBins == 2 * kSelThreads, "two bins per thread");
__device__ void find_bucket(SelSmem& sm, const uint32_t* h) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const uint32_t rem = sm.rem;               // rewritten only after the barriers below
  const uint32_t c0 = h[kBins - 1 - 2 * tid], c1 = h[kBins - 2 - 2 * tid], tot = c0 + c1;
  uint32_t x = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm.red[0][wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t s = sm.red[0][lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += y;
    }
    sm.red[0][lane] = s;
  }
  __syncthreads();
  const uint32_t before = (wid ? sm.red[0][wid - 1] : 0) + x - tot;
  if (before < rem && rem <= before + tot) {
    if (before + c0 >= rem) {
      sm.bucket = kBins - 1 - 2 * tid;
      sm.bucket_cnt = c0;
      sm.rem = rem - before;
    } else {
      sm.bucket = kBins - 2 - 2 * tid;
      sm.bucket_cnt = c1;
      sm.rem = rem - before - c0;
    }
  }
  __syncthreads();
}

// Lower edge (offset from the base key) of the final bucket: the first-pass
// bin b0 alone, or its refined sub-bin b1.
__device__ inline uint32_t pass_lo(uint32_t b0, int sh0, uint32_t b1, int width_shift, int sh1) {
  return width_shift == sh0 ? (b0 << sh0) : (b0 << sh0) + (b1 << sh1);
}

// Inverse of f32_key.
__device__ inline float key_f32(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Cluster-wide radix localisation of the k-th largest v key (keyU; 0 marks
// an invalid item).  kmin_l / kmax_l / dmax_l are this thread's minimum and
// maximum valid key and maximum delta.  The first pass spreads 2048 bins over
// the occupied key range; a second pass splits the chosen bin into 2048 more
// only when it holds more than kRefine items.  Returns muEdge >= the k-th
// largest U key and lamEdge <= the k-th largest L key (see the file comment).
constexpr uint32_t kRefine = 64;

__device__ void radix_edges(SelSmem& sm, const SelCtx& c, int n_local, uint32_t k, uint32_t kmin_l,
                            uint32_t kmax_l, float dmax_l, uint32_t& muEdge, uint32_t& lamEdge) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // ---- key range and the largest delta -------------------------------------------
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    kmin_l = min(kmin_l, __shfl_xor_sync(0xFFFFFFFFu, kmin_l, o));
    kmax_l = max(kmax_l, __shfl_xor_sync(0xFFFFFFFFu, kmax_l, o));
    dmax_l = fmaxf(dmax_l, __shfl_xor_sync(0xFFFFFFFFu, dmax_l, o));
  }
  if (lane == 0) { sm.red[0][wid] = kmin_l; sm.red[1][wid] = kmax_l; sm.dred[wid] = dmax_l; }
  __syncthreads();
  static_assert(kSelWarps == 32, "one lane per warp partial");
  // the key range and the largest bound, set by lane 0 of warp 0 (of rank 0's
  // view for a cluster: every rank computes the same values)
  auto set_range = [&](uint32_t lo, uint32_t hi, float dm) {
    sm.rem = k;
    sm.base_key = lo;
    sm.kmax_all = hi;
    sm.dmax_all = dm;
    const uint32_t range = hi - lo;
    const int bits = range ? 32 - __clz(range) : 0;
    sm.shift0 = bits > 11 ? bits - 11 : 0;
  };
  if (wid == 0) {                      // the warps' partials, one per lane
    uint32_t a0 = sm.red[0][lane], a1 = sm.red[1][lane];
    float dm = sm.dred[lane];
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      a0 = min(a0, __shfl_xor_sync(0xFFFFFFFFu, a0, o));
      a1 = max(a1, __shfl_xor_sync(0xFFFFFFFFu, a1, o));
      dm = fmaxf(dm, __shfl_xor_sync(0xFFFFFFFFu, dm, o));
    }
    if (lane == 0) {
      if (c.cs > 1) {
        sm.kmin = a0;
        sm.kmax = a1;
        sm.dmax = dm;
      } else {
        set_range(a0, a1, dm);
      }
    }
  }
  if (c.cs > 1) {
    cl_sync(c);
    if (wid == 0) {                    // the ranks' values, one rank per lane
      uint32_t a0 = 0xFFFFFFFFu, a1 = 0;
      float dm = 0.0f;
      if (lane < c.cs) {
        a0 = *remote(c, &sm.kmin, lane);
        a1 = *remote(c, &sm.kmax, lane);
        dm = *remote(c, &sm.dmax, lane);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        a0 = min(a0, __shfl_xor_sync(0xFFFFFFFFu, a0, o));
        a1 = max(a1, __shfl_xor_sync(0xFFFFFFFFu, a1, o));
        dm = fmaxf(dm, __shfl_xor_sync(0xFFFFFFFFu, dm, o));
      }
      if (lane == 0) set_range(a0, a1, dm);
    }
  }
  cl_sync(c);       // the range is read before any rank overwrites kmin / kmax
  const uint32_t kb = sm.base_key;
  const int sh0 = sm.shift0, sh1 = sh0 > 11 ? sh0 - 11 : 0;
  uint32_t b0 = 0;
  int width_shift = sh0;
  for (int pass = 0; pass < 2; ++pass) {
    for (int i = tid; i < kBins; i += blockDim.x) sm.hist[0][i] = 0;
    __syncthreads();
    const int sh = pass ? sh1 : sh0;
    for (int i = tid; i < n_local; i += blockDim.x) {
      const uint32_t u = sm.keyU[i];
      if (!u) continue;
      const uint32_t du = u - kb;
      if (pass == 0) atomicAdd(&sm.hist[0][du >> sh], 1u);
      else if ((du >> sh0) == b0) atomicAdd(&sm.hist[0][(du - (b0 << sh0)) >> sh], 1u);
    }
    cl_sync(c);
    const uint32_t* h = &sm.hist[0][0];
    if (c.cs > 1) {
      // the ranks' histograms summed: each rank sums its own slice of the bins
      // over the ranks (every rank's loads in flight together), then gathers
      // the other slices from their owners
      const int per = (kBins + c.cs - 1) / c.cs;
      const int lo = c.rank * per, hi = min(kBins, lo + per);
      for (int i = lo + tid; i < hi; i += blockDim.x) {
        uint32_t t = 0;
#pragma unroll 4
        for (int r = 0; r < kMaxSelCluster; ++r)
          if (r < c.cs) t += remote(c, &sm.hist[0][0], r)[i];
        sm.ghist[0][i] = t;
      }
      cl_sync(c);     // every slice summed; every rank has read every histogram before they are reset
      for (int i = tid; i < kBins; i += blockDim.x) {
        const int owner = i / per;
        if (owner != c.rank) sm.ghist[0][i] = remote(c, &sm.ghist[0][0], owner)[i];
      }
      __syncthreads();
      h = &sm.ghist[0][0];
    }
    find_bucket(sm, h);
    if (pass == 0) {
      b0 = sm.bucket;
      // narrow enough: few items, or a value width below the largest bound
      // (refining could not shrink the band by more than that)
      const uint64_t top = min64(int64_t(kb) + (int64_t(b0) << sh0) + ((int64_t(1) << sh0) - 1), int64_t(sm.kmax_all));
      const float wv = key_f32(uint32_t(top)) - key_f32(kb + (b0 << sh0));
      if (sh0 == 0 || sm.bucket_cnt <= kRefine || wv <= sm.dmax_all) break;
    } else {
      width_shift = sh1;
    }
  }
  const uint32_t lo = pass_lo(b0, sh0, sm.bucket, width_shift, sh1);
  // the bucket's top, clamped to the largest key (the k-th largest is below it)
  const uint64_t hi64 = uint64_t(kb) + lo + ((uint64_t(1) << width_shift) - 1);
  const uint32_t hi_key = hi64 > sm.kmax_all ? sm.kmax_all : uint32_t(hi64);
  const float D = sm.dmax_all;
  const float vlo = key_f32(kb + lo), vhi = key_f32(hi_key);
  muEdge = f32_key(__fadd_ru(vhi, D));
  lamEdge = f32_key(__fadd_rd(vlo, -D));
  __syncthreads();
}

// RN64(v * 2^e) for an int64 v, built with integer operations only (the
// fp64 conversion instructions are slow on this GPU).  Requires the result to
// be a normal fp64 number, which holds for every indexer product sum.
__device__ inline double int_to_f64_rn(long long v, int e) {
  if (v == 0) return 0.0;
  unsigned long long sign = v < 0 ? (1ull << 63) : 0ull;
  unsigned long long mag = v < 0 ? 0ull - (unsigned long long)v : (unsigned long long)v;
  int p = 63 - __clzll((long long)mag);          // leading bit index
  unsigned long long m;
  int ex = p + e;
  if (p <= 52) {
    m = mag << (52 - p);
  } else {
    int sh = p - 52;
    m = mag >> sh;
    unsigned long long rem = mag & ((1ull << sh) - 1), half = 1ull << (sh - 1);
    if (rem > half || (rem == half && (m & 1ull))) {
      ++m;
      if (m == (1ull << 53)) { m >>= 1; ++ex; }
    }
  }
  unsigned long long bits = sign | ((unsigned long long)(ex + 1023) << 52) | (m & ((1ull << 52) - 1));
  return __longlong_as_double((long long)bits);
}

// Exact fp64 value of an fp32 number, built with integer operations only.
__device__ inline double f32_to_f64_exact(float x) {
  uint32_t u = __float_as_uint(x);
  unsigned long long sign = (unsigned long long)(u >> 31) << 63;
  int E = (u >> 23) & 0xFF;
  uint32_t m = u & 0x7FFFFF;
  if (E == 0) {
    if (m == 0) return __longlong_as_double((long long)sign);
    int p = 31 - __clz(m);                       // subnormal: normalise
    unsigned long long mm = (unsigned long long)(m << (23 - p)) & 0x7FFFFF;
    int ex = p - 149;
    return __longlong_as_double((long long)(sign | ((unsigned long long)(ex + 1023) << 52) | (mm << 29)));
  }
  return __longlong_as_double((long long)(sign | ((unsigned long long)(E - 127 + 1023) << 52) |
                                          ((unsigned long long)m << 29)));
}

struct ItemVal {
  float v, delta;
  bool valid;
};

__device__ inline ItemVal load_item(const IdxArgs& a, ItemKind kind, const SelCtx& c,
                                    const int32_t* pool_ids, int64_t item) {
  const float* __restrict__ ws_f = reinterpret_cast<const float*>(a.ws);
  ItemVal r = {0.0f, 0.0f, false};
  if (kind == kBlocks) {
    int64_t nb = (c.n_ctx + kBlock - 1) / kBlock;
    if (item < nb) {
      r.valid = true;
      r.v = ws_f[(a.L.blk_scores >> 2) + int64_t(c.b) * a.L.nb_max + item];
      r.delta = ws_f[(a.L.blk_delta >> 2) + int64_t(c.b) * a.L.nb_max + item];
    }
  } else {
    int32_t blk = pool_ids[item >> 3];
    int64_t t = int64_t(blk) * kBlock + (item & 7);
    if (blk >= 0 && t < c.n_ctx) {
      r.valid = true;
      if (kind == kPoolPos) {
        r.v = ws_f[(a.L.pos_scores >> 2) + int64_t(c.b) * a.d.max_ctx + t];
        r.delta = ws_f[(a.L.blk_delta >> 2) + int64_t(c.b) * a.L.nb_max + blk];
      } else {
        int64_t P8 = int64_t(a.d.pool_blocks) * kBlock;
        r.v = ws_f[(a.L.ri_scores >> 2) + int64_t(c.b) * P8 + item];
        r.delta = ws_f[(a.L.ri_delta >> 2) + int64_t(c.b) * a.d.pool_blocks + (item >> 3)];
      }
    }
  }
  return r;
}

// Exact scores of a list of positions (fp64, -inf for invalid ones), using
// the whole CTA, in rounds of up to kExRows positions.  In round r the first
// kExSumThreads threads form the ordered fp64 head sums of round r - 1 (a
// chain of dependent fp64 additions, one thread per position) while the
// other threads stage round r's indexer-K rows in shared memory and compute
// its products w_h * ReLU(d_h): one thread per (position, head) sums the Di
// exact products serially in int64, in a 128-bit integer when their span is
// wider (the usual case for fp32 keys), or in the multi-limb accumulator
// beyond 126 bits, and rounds once.
__device__ void exact_scores(const IdxArgs& a, SelSmem& sm, const SelCtx& c, const int64_t* pos,
                             int np, double* out) {
  ExScratch& ex = ex_scratch(sm);
  const int tid = threadIdx.x;
  const int hi = a.d.idx_heads, di = a.d.idx_dim;
  const bool fp8 = a.d.idx_k_dtype == CSA2_IDXK_E4M3;
  const int rounds = (np + kExRows - 1) / kExRows;
  constexpr int kWork = kSelThreads - kExSumThreads;
  for (int r = 0; r <= rounds; ++r) {
    if (tid < kExSumThreads) {
      // ---- ordered head sums of the previous round --------------------------------
      if (r > 0) {
        const int r0 = (r - 1) * kExRows, nr = min(kExRows, np - r0);
        if (tid < nr) {
          const int64_t t = pos[r0 + tid];
          double sum = -INFINITY;
          if (t >= 0 && t < c.n_ctx) {
            sum = 0.0;
            const double* row = ex.dd[(r - 1) & 1] + tid * kMaxIdxHeads;
            for (int h = 0; h < hi; ++h) sum = __dadd_rn(sum, row[h]);
          }
          out[r0 + tid] = sum;
        }
      }
    } else if (r < rounds) {
      const int wt = tid - kExSumThreads;
      const int r0 = r * kExRows, nr = min(kExRows, np - r0);
      // ---- stage the rows: E4M3 keys as exact integers k * 2^9, fp32 keys as
      //      bits; 4-byte words of the rows, every load of a batch issued first
      const int wpr = fp8 ? di >> 2 : di;            // words of a row
      for (int w0 = 0; w0 < nr * wpr; w0 += kStageWords * kWork) {
        int64_t srow[kStageWords];
        uint32_t sw[kStageWords];
#pragma unroll
        for (int j = 0; j < kStageWords; ++j) {
          const int i = w0 + wt + j * kWork;
          srow[j] = -1;
          if (i < nr * wpr) {
            const int64_t t = pos[r0 + i / wpr];
            if (t >= 0 && t < c.n_ctx) srow[j] = kv_row(a.page_table, a.d, c.b, t, a.ws);
          }
        }
#pragma unroll
        for (int j = 0; j < kStageWords; ++j) {
          const int i = w0 + wt + j * kWork;
          sw[j] = srow[j] >= 0 ? reinterpret_cast<const uint32_t*>(a.idx_k)[srow[j] * wpr + i % wpr] : 0u;
        }
#pragma unroll
        for (int j = 0; j < kStageWords; ++j) {
          const int i = w0 + wt + j * kWork;
          if (i >= nr * wpr) break;
          int32_t* dst = ex.krows + (i / wpr) * kExRowWords;
          if (fp8) {
            int32_t kq[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const Factor f = factor_e4m3((sw[j] >> (8 * q)) & 0xFFu);
              kq[q] = f.sig * (1 << (f.exp + 9));
            }
            reinterpret_cast<int4*>(dst)[i % wpr] = make_int4(kq[0], kq[1], kq[2], kq[3]);
          } else {
            dst[i % wpr] = int32_t(sw[j]);
          }
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kWork) : "memory");
      // ---- products of this round --------------------------------------------------
      for (int task = wt; task < nr * hi; task += kWork) {
        const int rr = task / hi, h = task % hi;
        const int32_t* kr = ex.krows + rr * kExRowWords;
        double d;
        if (fp8 && sm.q_fast[h]) {
          // |sum| <= sum|qi| * 448*2^9 < 2^62: the int64 sum is exact
          // 16-byte loads of 4 channels of the query row and of the key row
          const int4* q4 = reinterpret_cast<const int4*>(sm.qi + h * kQiStride);
          const int4* k4 = reinterpret_cast<const int4*>(kr);
          long long acc = 0;
#pragma unroll 8
          for (int c4 = 0; c4 < 32; ++c4) {
            const int4 qv = q4[c4], kv = k4[c4];
            acc += (long long)qv.x * kv.x;
            acc += (long long)qv.y * kv.y;
            acc += (long long)qv.z * kv.z;
            acc += (long long)qv.w * kv.w;
          }
          d = int_to_f64_rn(acc, sm.q_elo[h] - 9);
        } else {
          auto kf = [&](int ch) {
            return fp8 ? Factor{kr[ch], -9} : factor_f32(__int_as_float(kr[ch]));
          };
          d = exact_head_dot([&](int ch) { return sm.qf[ch * kMaxIdxHeads + h]; }, di, kf);
        }
        // w_h * ReLU(d_h)
        const unsigned long long db = (unsigned long long)__double_as_longlong(d);
        const bool positive = (db >> 63) == 0 && db != 0;
        ex.dd[r & 1][rr * kMaxIdxHeads + h] = __dmul_rn(f32_to_f64_exact(sm.w[h]), positive ? d : 0.0);
      }
    }
    __syncthreads();
  }
}

static_assert(kFastRows * 128 <= int(sizeof(int32_t)) * kExRows * kExRowWords, "staged FP4 rows fit");
static_assert(kFastRows * kMaxIdxHeads <= 2 * kExRows * kMaxIdxHeads, "head products fit");

// FP4 query and keys: d_h = sum_g sk_g sq_hg I_hg / 4 with I_hg = sum over the
// group of (2 qhat)(2 khat), small integers.  Writing each E4M3 scale as
// M 2^E (M <= 15, E in [-9, 5]), the group term times 2^20 is the integer
// M_k M_q I << (E_k + E_q + 18) (shift 0..28, below 2^47); the 8 terms sum
// exactly in int64 (below 2^50) and d_h = sum * 2^-20 is exact in fp64.
// Staging: 8 threads per position, one group each (8 code bytes widened to
// 16 signed bytes, and the scale's M, E); products: one thread per
// (position, head), its 8 groups (dp4a).
__device__ void exact_scores_fp4(const IdxArgs& a, SelSmem& sm, const SelCtx& c, const int64_t* pos, int np,
                                 double* out) {
  ExScratch& ex = ex_scratch(sm);
  const int tid = threadIdx.x, hi = a.d.idx_heads;
  uint4* rows = reinterpret_cast<uint4*>(ex.krows);           // [kFastRows][8] x 16 signed bytes
  int2* ksc = reinterpret_cast<int2*>(ex.krows + kFastRows * 32);   // [kFastRows][8] (M, E)
  double* dd = &ex.dd[0][0];                                   // [kFastRows][kMaxIdxHeads]
  if (tid < np * 8) {
    const int p = tid >> 3, g = tid & 7;
    const int64_t t = pos[p];
    uint2 cw = make_uint2(0, 0);
    uint32_t sc = 0;
    if (t >= 0 && t < c.n_ctx) {
      const int64_t r = kv_row(a.page_table, a.d, c.b, t, a.ws);
      if (r >= 0) {
        cw = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(a.idx_k) + r * 64) + g);
        sc = __ldg(a.idx_scales + r * 8 + g);
      }
    }
    rows[p * 8 + g] = make_uint4(e2m1x4_to_i8x4_twice(cw.x), e2m1x4_to_i8x4_twice(cw.x >> 16),
                                 e2m1x4_to_i8x4_twice(cw.y), e2m1x4_to_i8x4_twice(cw.y >> 16));
    const Factor f = factor_e4m3(sc);
    ksc[p * 8 + g] = make_int2(f.sig, f.exp);
  }
  __syncthreads();
  // one thread per (position, head): its 8 group terms, the dot rounded once
  // to fp64 and w_h * ReLU(d_h) (the fp64 steps in full warps)
  for (int i = tid; i < np * hi; i += kSelThreads) {
    const int p = i / hi, h = i - p * hi;
    const uint4* q4 = reinterpret_cast<const uint4*>(sm.qi + h * kQiStride);
    long long acc = 0;
#pragma unroll 2
    for (int g = 0; g < 8; ++g) {
      const uint4 kv = rows[p * 8 + g], qv = q4[g];
      int dot = __dp4a(int(kv.x), int(qv.x), 0);
      dot = __dp4a(int(kv.y), int(qv.y), dot);
      dot = __dp4a(int(kv.z), int(qv.z), dot);
      dot = __dp4a(int(kv.w), int(qv.w), dot);
      const int2 kf = ksc[p * 8 + g];
      const Factor qf = sm.qf[h * 8 + g];
      acc += (long long)(kf.x * qf.sig * dot) * (1ll << (kf.y + qf.exp + 18));   // shift 0..28
    }
    const double d = int_to_f64_rn(acc, -20);
    const unsigned long long db = (unsigned long long)__double_as_longlong(d);
    const bool positive = (db >> 63) == 0 && db != 0;
    dd[p * kMaxIdxHeads + h] = __dmul_rn(f32_to_f64_exact(sm.w[h]), positive ? d : 0.0);
  }
  __syncthreads();
  if (tid < np) {
    const int64_t t = pos[tid];
    double sum = -INFINITY;
    if (t >= 0 && t < c.n_ctx) {
      sum = 0.0;
      for (int h = 0; h < hi; ++h) sum = __dadd_rn(sum, dd[tid * kMaxIdxHeads + h]);
    }
    out[tid] = sum;
  }
  __syncthreads();
}

// Exact scores of up to kFastRows positions in one pass (E4M3 keys, every
// head's query on the int64 path).  The positions' key rows are staged once
// as the integers k*2^9 (all loads in flight together).  Then one thread per
// (position, head) sums its 128 exact products k*2^9 x qi in int64 (a warp's
// 32 pairs read one or two staged rows and the rows of up to 16 heads of the
// integer query: broadcasts, no cross-lane reduction), rounds the dot once to
// fp64 and forms w_h * ReLU(d_h); one thread per position adds the heads in
// order in fp64.  -inf for invalid positions.
__device__ void exact_scores_fast(const IdxArgs& a, SelSmem& sm, const SelCtx& c, const int64_t* pos, int np,
                                  double* out) {
  ExScratch& ex = ex_scratch(sm);
  const int tid = threadIdx.x, hi = a.d.idx_heads;
  double* dd = &ex.dd[0][0];                                   // [kFastRows][kMaxIdxHeads]
  int32_t* kdec = reinterpret_cast<int32_t*>(dd + kFastRows * kMaxIdxHeads);   // [kFastRows][128]
  // ---- stage the rows: 8 threads per position, the words 8j + e of the row ----
  if (tid < np * 8) {
    const int p = tid >> 3, e = tid & 7;
    const int64_t t = pos[p];
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (t >= 0 && t < c.n_ctx) {
      const int64_t r = kv_row(a.page_table, a.d, c.b, t, a.ws);
      if (r >= 0) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(a.idx_k) + r * 128) + e;
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = __ldg(src + 8 * j);
      }
    }
    int4* dst = reinterpret_cast<int4*>(kdec + p * 128) + e;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      dst[8 * j] = make_int4(sm.k_lut[w[j] & 0xFF], sm.k_lut[(w[j] >> 8) & 0xFF], sm.k_lut[(w[j] >> 16) & 0xFF],
                             sm.k_lut[w[j] >> 24]);
  }
  __syncthreads();
  // ---- one (position, head) per thread: the exact dot, then w_h * ReLU(d_h) -------
  for (int i = tid; i < np * hi; i += kSelThreads) {
    const int p = i / hi, h = i - p * hi;
    const int4* kr = reinterpret_cast<const int4*>(kdec + p * 128);
    const int4* qr = reinterpret_cast<const int4*>(sm.qi + h * kQiStride);
    long long acc0 = 0, acc1 = 0;                              // two chains, summed exactly
#pragma unroll 2
    for (int c4 = 0; c4 < 32; c4 += 2) {
      const int4 k0 = kr[c4], q0 = qr[c4], k1 = kr[c4 + 1], q1 = qr[c4 + 1];
      acc0 += (long long)q0.x * k0.x;
      acc1 += (long long)q1.x * k1.x;
      acc0 += (long long)q0.y * k0.y;
      acc1 += (long long)q1.y * k1.y;
      acc0 += (long long)q0.z * k0.z;
      acc1 += (long long)q1.z * k1.z;
      acc0 += (long long)q0.w * k0.w;
      acc1 += (long long)q1.w * k1.w;
    }
    const double d = int_to_f64_rn(acc0 + acc1, sm.q_elo[h] - 9);
    const unsigned long long db = (unsigned long long)__double_as_longlong(d);
    const bool positive = (db >> 63) == 0 && db != 0;
    dd[p * kMaxIdxHeads + h] = __dmul_rn(f32_to_f64_exact(sm.w[h]), positive ? d : 0.0);
  }
  __syncthreads();
  // ---- ordered head sums ----------------------------------------------------------
  if (tid < np) {
    const int64_t t = pos[tid];
    double sum = -INFINITY;
    if (t >= 0 && t < c.n_ctx) {
      sum = 0.0;
      for (int h2 = 0; h2 < hi; ++h2) sum = __dadd_rn(sum, dd[tid * kMaxIdxHeads + h2]);
    }
    out[tid] = sum;
  }
  __syncthreads();
}

// Monotone 64-bit key of a double (larger value -> larger key).
__device__ inline uint64_t f64_key(double x) {
  uint64_t u = uint64_t(__double_as_longlong(x + 0.0));
  return (u >> 63) ? ~u : (u | (uint64_t(1) << 63));
}

// Selects the k best of n items of `kind`; writes their ids ascending to
// out[0 .. k).  All CTAs of the cluster take part (items split by rank).
// With `superset` (block items) no exact re-scoring takes place: the ids of
// every item whose bounds let it be among the k best (the certain ones and the
// band) are written ascending, at most pool_blocks of them.  Returns the
// number of items selected (superset: all of them, also those not written).
template <bool kFp4>
__device__ int64_t certified_select(const IdxArgs& a, SelSmem& sm, const SelCtx& c, ItemKind kind,
                                    int64_t n_items, int64_t k, int32_t* out, bool superset = false) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // the items are split evenly over the cluster's CTAs (whole 32-item words)
  const int64_t per = min64(kSelCapPerCta, ((n_items + c.cs - 1) / c.cs + 31) & ~int64_t(31));
  const int64_t base = int64_t(c.rank) * per;
  const int n_local = int(max64(0, min64(per, n_items - base)));
  const int nwords = (n_local + 31) / 32;
  for (int i = tid; i < kSelCapPerCta / 32; i += blockDim.x) { sm.band_bits[i] = 0; sm.sel_bits[i] = 0; }
  if (tid == 0) { sm.cnt_in = 0; sm.cnt_band = 0; }
  __syncthreads();
  uint32_t kmin_l = 0xFFFFFFFFu, kmax_l = 0;
  float dmax_l = 0.0f;
  if (kind != kBlocks) {
    // positions: the 8 items of a pool block are contiguous scores with one
    // bound; a thread takes whole blocks (2 per thread at most)
    const float* ws_f = reinterpret_cast<const float*>(a.ws);
    const bool vec = kind == kReindexPos || (a.d.max_ctx & 7) == 0;   // 32-byte aligned blocks in the row
    constexpr int kPB = kSelCapPerCta / kBlock / kSelThreads;   // blocks per thread
    // every load of this thread is issued before any key is formed
    float v[kPB][kBlock], dl[kPB];
    int nv[kPB];                                     // valid positions of the block
#pragma unroll
    for (int k = 0; k < kPB; ++k) {
      const int jb = tid + k * kSelThreads;
      const int64_t gi0 = base + int64_t(jb) * kBlock;
      dl[k] = -1.0f;
      nv[k] = 0;
#pragma unroll
      for (int i = 0; i < kBlock; ++i) v[k][i] = 0.0f;
      if (jb * kBlock >= n_local) continue;
      const int32_t blk = sm.pool_ids[gi0 >> 3];
      if (blk >= 0 && int64_t(blk) * kBlock < c.n_ctx) {
        nv[k] = int(min64(kBlock, c.n_ctx - int64_t(blk) * kBlock));
        const float* src;
        if (kind == kPoolPos) {
          src = ws_f + (a.L.pos_scores >> 2) + int64_t(c.b) * a.d.max_ctx + int64_t(blk) * kBlock;
          dl[k] = ws_f[(a.L.blk_delta >> 2) + int64_t(c.b) * a.L.nb_max + blk];
        } else {
          src = ws_f + (a.L.ri_scores >> 2) + int64_t(c.b) * a.d.pool_blocks * kBlock + gi0;
          dl[k] = ws_f[(a.L.ri_delta >> 2) + int64_t(c.b) * a.d.pool_blocks + (gi0 >> 3)];
        }
        if (vec) {
          const float4 lo = reinterpret_cast<const float4*>(src)[0], hi = reinterpret_cast<const float4*>(src)[1];
          v[k][0] = lo.x; v[k][1] = lo.y; v[k][2] = lo.z; v[k][3] = lo.w;
          v[k][4] = hi.x; v[k][5] = hi.y; v[k][6] = hi.z; v[k][7] = hi.w;
        } else {
#pragma unroll
          for (int i = 0; i < kBlock; ++i) v[k][i] = i < nv[k] ? src[i] : 0.0f;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kPB; ++k) {
      const int jb = tid + k * kSelThreads;
      if (jb * kBlock >= n_local) break;
      uint32_t kv[kBlock], kd[kBlock];
#pragma unroll
      for (int i = 0; i < kBlock; ++i) {
        kv[i] = 0;
        kd[i] = 0;
        if (i < nv[k]) {
          kv[i] = f32_key(v[k][i]);
          kd[i] = __float_as_uint(dl[k]);
          kmin_l = min(kmin_l, kv[i]);
          kmax_l = max(kmax_l, kv[i]);
          dmax_l = fmaxf(dmax_l, dl[k]);
        }
      }
      uint4* ku = reinterpret_cast<uint4*>(sm.keyU + jb * kBlock);
      uint4* kl = reinterpret_cast<uint4*>(sm.keyL + jb * kBlock);
      ku[0] = make_uint4(kv[0], kv[1], kv[2], kv[3]);
      ku[1] = make_uint4(kv[4], kv[5], kv[6], kv[7]);
      kl[0] = make_uint4(kd[0], kd[1], kd[2], kd[3]);
      kl[1] = make_uint4(kd[4], kd[5], kd[6], kd[7]);
    }
  } else {
    // every item load of this thread is issued before any key is formed
    constexpr int kPer = kSelCapPerCta / kSelThreads;
    float vv[kPer], dd[kPer];                        // dd < 0: not an item
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = tid + j * kSelThreads;
      const ItemVal it = i < n_local ? load_item(a, kind, c, sm.pool_ids, base + i) : ItemVal{0.0f, 0.0f, false};
      vv[j] = it.v;
      dd[j] = it.valid ? it.delta : -1.0f;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = tid + j * kSelThreads;
      if (i >= n_local) break;
      uint32_t kv = 0, kd = 0;
      if (dd[j] >= 0.0f) {
        kv = f32_key(vv[j]);
        kd = __float_as_uint(dd[j]);
        kmin_l = min(kmin_l, kv);
        kmax_l = max(kmax_l, kv);
        dmax_l = fmaxf(dmax_l, dd[j]);
      }
      sm.keyU[i] = kv;                               // v key (0: not an item)
      sm.keyL[i] = kd;                               // delta bits
    }
  }
  __syncthreads();
  // The 32 items of a word are one warp's in each pass over the items: the
  // warp forms the word by ballot and lane 0 stores it (no shared atomics).
  if (k >= n_items) {
    for (int i0 = tid - lane; i0 < n_local; i0 += blockDim.x) {
      const int i = i0 + lane;
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, i < n_local && sm.keyU[i] != 0);
      if (lane == 0) sm.sel_bits[i0 >> 5] = m;
    }
  } else {
    uint32_t muE, lamE;
    radix_edges(sm, c, n_local, uint32_t(k), kmin_l, kmax_l, dmax_l, muE, lamE);
    uint32_t my_in = 0, my_band = 0;                  // lane 0's warp totals
    // key order is float order (-0 and +0 one key): compare the bounds as floats
    const float muF = key_f32(muE), lamF = key_f32(lamE);
    if (superset) {
      // every item that may be among the k best (certain or in the band): U >= lambda'
      for (int i0 = tid - lane; i0 < n_local; i0 += blockDim.x) {
        const int i = i0 + lane;
        const uint32_t kv = i < n_local ? sm.keyU[i] : 0u;
        const bool may = kv != 0 && __fadd_ru(key_f32(kv), __uint_as_float(sm.keyL[i])) >= lamF;
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, may);
        if (lane == 0) sm.sel_bits[i0 >> 5] = m;
      }
    } else {
      for (int i0 = tid - lane; i0 < n_local; i0 += blockDim.x) {
        const int i = i0 + lane;
        const uint32_t kv = i < n_local ? sm.keyU[i] : 0u;
        bool in = false, band = false;
        if (kv != 0) {
          const float v = key_f32(kv), dl = __uint_as_float(sm.keyL[i]);
          in = __fadd_rd(v, -dl) > muF;
          band = !in && __fadd_ru(v, dl) >= lamF;
        }
        const uint32_t mi = __ballot_sync(0xFFFFFFFFu, in), mb = __ballot_sync(0xFFFFFFFFu, band);
        if (lane == 0) {
          sm.sel_bits[i0 >> 5] = mi;
          sm.band_bits[i0 >> 5] = mb;
          my_in += __popc(mi);
          my_band += __popc(mb);
        }
      }
      if (lane == 0) {
        atomicAdd(&sm.cnt_in, my_in);
        atomicAdd(&sm.cnt_band, my_band);
      }
      // this side's band scratch in the workspace (cluster case, large bands)
      const int64_t wso = (int64_t(c.b) * 2 + c.side) * a.L.sel_cap;
      double* g_exact = reinterpret_cast<double*>(a.ws + a.L.sel_exact) + wso;
      int32_t* g_list = reinterpret_cast<int32_t*>(a.ws + a.L.sel_list) + wso;
      uint8_t* g_pick = a.ws + a.L.sel_pick + wso;
      // ordered list of this CTA's band items (keyL area is free now)
      uint32_t nband = scan_words(sm, sm.band_bits, nwords);
      int32_t* blist = reinterpret_cast<int32_t*>(sm.keyL);
      for (int wv = tid; wv < nwords; wv += blockDim.x) {
        uint32_t bits = sm.band_bits[wv], o = sm.word_off[wv];
        while (bits) {
          int bp = __ffs(bits) - 1;
          bits &= bits - 1;
          blist[o++] = wv * 32 + bp;
        }
      }
      __syncthreads();
      // A selection held by one CTA with a band of at most kSelThreads items
      // keeps the band's exact-score keys in shared memory (in the histogram
      // space, free after the radix step) and marks its picks directly; the
      // workspace lists serve the cluster case and larger bands.
      const bool local_pick = c.cs == 1 && nband <= uint32_t(kSelThreads);
      uint64_t* band_key = reinterpret_cast<uint64_t*>(&sm.hist[0][0]);
      static_assert(sizeof(sm.hist) >= kSelThreads * sizeof(uint64_t), "band keys fit the histograms");
      // exact scores of the band, a chunk of items at a time.  For a block,
      // only the positions whose upper bound reaches the block's best lower
      // bound can hold its exact maximum; the others are not re-scored.
      const float* ws_f = reinterpret_cast<const float*>(a.ws);
      ExScratch& ex = ex_scratch(sm);
      for (uint32_t j0 = 0; j0 < nband; j0 += kExItems) {
        const int nit = int(min64(kExItems, int64_t(nband) - j0));
        if (tid == 0) sm.n_cand = 0;
        __syncthreads();
        // a few band blocks: every valid position of each is a candidate (no
        // filter by the position scores, one round trip less)
        const bool all_pos = sm.fast_exact && kind == kBlocks && nit * kBlock <= kFastRows;
        if (all_pos) {
          if (tid < nit * kBlock) {
            const int j = tid >> 3;
            const int64_t t = (base + blist[j0 + j]) * kBlock + (tid & 7);
            ex.cand_pos[tid] = t < c.n_ctx ? t : -1;
            ex.cand_item[tid] = j;
            if ((tid & 7) == 0) ex.item_best[j] = 0;
          }
          if (tid == 0) sm.n_cand = uint32_t(nit * kBlock);
        }
        for (int j = all_pos ? nit : wid; j < nit; j += kSelWarps) {
          int64_t gi = base + blist[j0 + j];
          if (kind == kBlocks) {
            int64_t t = gi * kBlock + (lane & 7);
            bool ok = lane < kBlock && t < c.n_ctx;
            float dl = ws_f[(a.L.blk_delta >> 2) + int64_t(c.b) * a.L.nb_max + gi];
            float v = ok ? ws_f[(a.L.pos_scores >> 2) + int64_t(c.b) * a.d.max_ctx + t] : -INFINITY;
            float lo = ok ? __fadd_rd(v, -dl) : -INFINITY;
            float hv = ok ? __fadd_ru(v, dl) : -INFINITY;
            float lmax = lo;
  #pragma unroll
            for (int o = 16; o; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
            bool cand = ok && hv >= lmax;
            uint32_t m = __ballot_sync(0xFFFFFFFFu, cand);
            uint32_t slot0 = 0;
            if (lane == 0) slot0 = atomicAdd(&sm.n_cand, uint32_t(__popc(m)));
            slot0 = __shfl_sync(0xFFFFFFFFu, slot0, 0);
            if (cand) {
              uint32_t sl = slot0 + __popc(m & ((1u << lane) - 1));
              ex.cand_pos[sl] = t;
              ex.cand_item[sl] = j;
            }
          } else if (lane == 0) {
            int32_t blk = sm.pool_ids[gi >> 3];
            uint32_t sl = atomicAdd(&sm.n_cand, 1u);
            ex.cand_pos[sl] = blk < 0 ? -1 : int64_t(blk) * kBlock + (gi & 7);
            ex.cand_item[sl] = j;
          }
          if (lane == 0) ex.item_best[j] = 0;       // key of -inf is above 0
        }
        __syncthreads();
        const int ncand = int(sm.n_cand);
        if constexpr (kFp4) {
          for (int c0 = 0; c0 < ncand; c0 += kFastRows)
            exact_scores_fp4(a, sm, c, ex.cand_pos + c0, min(kFastRows, ncand - c0), ex.cand_score + c0);
        } else if (sm.fast_exact) {
          for (int c0 = 0; c0 < ncand; c0 += kFastRows)
            exact_scores_fast(a, sm, c, ex.cand_pos + c0, min(kFastRows, ncand - c0), ex.cand_score + c0);
        } else {
          exact_scores(a, sm, c, ex.cand_pos, ncand, ex.cand_score);
        }
        for (int i = tid; i < ncand; i += blockDim.x)
          atomicMax(&ex.item_best[ex.cand_item[i]], f64_key(ex.cand_score[i]));
        __syncthreads();
        for (int j = tid; j < nit; j += blockDim.x) {
          int64_t gi = base + blist[j0 + j];
          uint64_t kk = ex.item_best[j];
          if (local_pick) {
            band_key[j0 + j] = kk ? kk : f64_key(-INFINITY);   // the key of the decoded score
            continue;
          }
          uint64_t u = (kk >> 63) ? (kk & ~(uint64_t(1) << 63)) : ~kk;   // inverse of f64_key
          g_exact[gi] = kk ? __longlong_as_double((long long)u) : -INFINITY;
          g_pick[gi] = 0;
        }
        __syncthreads();
      }
      cl_sync(c);
      uint32_t tot_in = sm.cnt_in, tot_band = sm.cnt_band, band_off = 0;
      if (c.cs > 1) {
        // the ranks' counters, one rank per lane of warp 0 (not one remote read
        // per rank by every thread)
        if (wid == 0) {
          uint32_t ci = 0, cb = 0;
          if (lane < c.cs) {
            ci = *remote(c, &sm.cnt_in, lane);
            cb = *remote(c, &sm.cnt_band, lane);
          }
          const uint32_t ti = __reduce_add_sync(0xFFFFFFFFu, ci), tb = __reduce_add_sync(0xFFFFFFFFu, cb);
          const uint32_t bo = __reduce_add_sync(0xFFFFFFFFu, lane < c.rank ? cb : 0u);
          if (lane == 0) { sm.tot3[0] = ti; sm.tot3[1] = tb; sm.tot3[2] = bo; }
        }
        __syncthreads();
        tot_in = sm.tot3[0];
        tot_band = sm.tot3[1];
        band_off = sm.tot3[2];
      }
      if (!local_pick)
        for (uint32_t j = tid; j < nband; j += blockDim.x) g_list[band_off + j] = int32_t(base + blist[j]);
      cl_sync(c);
      // ---- rank 0 picks the best (k - tot_in) band items by exact score -----
      int64_t need = k - int64_t(tot_in);
      if (c.rank == 0 && need > 0) {
        if (need >= int64_t(tot_band)) {
          for (uint32_t i = tid; i < tot_band; i += blockDim.x) {
            if (local_pick) atomicOr(&sm.sel_bits[blist[i] >> 5], 1u << (blist[i] & 31));
            else g_pick[g_list[i]] = 1;
          }
        } else if (tot_band <= kSelThreads) {
          // small band: each item's rank = the number of band items ahead of it
          uint64_t* skey = reinterpret_cast<uint64_t*>(sm.keyU);
          int32_t* sidx = reinterpret_cast<int32_t*>(sm.keyL);
          for (uint32_t i = tid; i < tot_band; i += blockDim.x) {
            if (local_pick) {                    // sidx is the band list itself (base 0)
              skey[i] = band_key[i];
            } else {
              int32_t it = g_list[i];
              skey[i] = f64_key(g_exact[it]);
              sidx[i] = it;
            }
          }
          __syncthreads();
          // one warp per item: the lanes count the band items ahead of it
          for (uint32_t i = wid; i < tot_band; i += kSelWarps) {
            const uint64_t mk = skey[i];
            const int32_t mi = sidx[i];
            uint32_t rank = 0;
            for (uint32_t j = lane; j < tot_band; j += 32) {
              const uint64_t kj = skey[j];
              rank += (kj > mk || (kj == mk && sidx[j] < mi)) ? 1u : 0u;
            }
            rank = __reduce_add_sync(0xFFFFFFFFu, rank);
            if (lane == 0 && rank < uint32_t(need)) {
              if (local_pick) atomicOr(&sm.sel_bits[mi >> 5], 1u << (mi & 31));
              else g_pick[mi] = 1;
            }
          }
        } else if (tot_band <= kSortCap) {
          uint64_t* skey = reinterpret_cast<uint64_t*>(sm.keyU);
          int32_t* sidx = reinterpret_cast<int32_t*>(sm.keyL);
          int nsort = 1;
          while (nsort < int(tot_band)) nsort <<= 1;
          for (int i = tid; i < nsort; i += blockDim.x) {
            if (i < int(tot_band)) { int32_t it = g_list[i]; skey[i] = f64_key(g_exact[it]); sidx[i] = it; }
            else { skey[i] = 0; sidx[i] = INT_MAX; }
          }
          __syncthreads();
          for (int size = 2; size <= nsort; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
              for (int i = tid; i < nsort; i += blockDim.x) {
                int j = i ^ stride;
                if (j > i) {
                  bool desc = (i & size) == 0;
                  bool i_first = skey[i] > skey[j] || (skey[i] == skey[j] && sidx[i] < sidx[j]);
                  if (desc != i_first) {
                    uint64_t tk = skey[i]; skey[i] = skey[j]; skey[j] = tk;
                    int32_t ti = sidx[i]; sidx[i] = sidx[j]; sidx[j] = ti;
                  }
                }
              }
              __syncthreads();
            }
          }
          for (int i = tid; i < need; i += blockDim.x) g_pick[sidx[i]] = 1;
        } else {
          // large band (massive exact ties): 64-bit radix select streamed over
          // the global band list by this CTA alone
          uint32_t* h64 = &sm.hist[0][0];
          __shared__ unsigned long long pref64;
          __shared__ uint32_t rem64;
          if (tid == 0) { pref64 = 0; rem64 = uint32_t(need); }
          __syncthreads();
          for (int pass = 0; pass < 8; ++pass) {
            int shift = 56 - 8 * pass;
            uint64_t maskHi = pass ? (~uint64_t(0) << (64 - 8 * pass)) : 0;
            if (tid < 256) h64[tid] = 0;
            __syncthreads();
            for (uint32_t i = tid; i < tot_band; i += blockDim.x) {
              uint64_t key = f64_key(g_exact[g_list[i]]);
              if ((key & maskHi) == pref64) atomicAdd(&h64[(key >> shift) & 0xFF], 1u);
            }
            __syncthreads();
            if (tid == 0) {
              uint32_t acc = 0;
              for (int bkt = 255; bkt >= 0; --bkt) {
                if (acc + h64[bkt] >= rem64) { pref64 |= uint64_t(bkt) << shift; rem64 -= acc; break; }
                acc += h64[bkt];
              }
            }
            __syncthreads();
          }
          if (tid == 0) {
            uint64_t kappa = pref64;
            uint32_t taken = 0;
            for (uint32_t i = 0; i < tot_band; ++i) {
              uint64_t key = f64_key(g_exact[g_list[i]]);
              if (key > kappa) g_pick[g_list[i]] = 1;
              else if (key == kappa && taken < rem64) { g_pick[g_list[i]] = 1; ++taken; }
            }
          }
        }
      }
      cl_sync(c);
      if (!local_pick)
        for (int wv = tid; wv < nwords; wv += blockDim.x) {
          uint32_t bits = sm.band_bits[wv];
          while (bits) {
            int bp = __ffs(bits) - 1;
            bits &= bits - 1;
            if (g_pick[base + wv * 32 + bp]) atomicOr(&sm.sel_bits[wv], 1u << bp);
          }
        }
    }
  }
  // ---- ordered output ------------------------------------------------------
  uint32_t nsel = scan_words(sm, sm.sel_bits, nwords);
  if (tid == 0) sm.cnt_sel = nsel;
  cl_sync(c);
  uint32_t off = 0;
  int64_t total = nsel;
  if (c.cs > 1) {
    if (wid == 0) {
      const uint32_t mine = lane < c.cs ? *remote(c, &sm.cnt_sel, lane) : 0u;
      const uint32_t v = __reduce_add_sync(0xFFFFFFFFu, lane < c.rank ? mine : 0u);
      const uint32_t all = __reduce_add_sync(0xFFFFFFFFu, mine);
      if (lane == 0) { sm.tot3[0] = v; sm.tot3[1] = all; }
    }
    __syncthreads();
    off = sm.tot3[0];
    total = sm.tot3[1];
  }
  const int64_t cap = superset ? int64_t(a.d.pool_blocks) : k;
  for (int wv = tid; wv < nwords; wv += blockDim.x) {
    uint32_t bits = sm.sel_bits[wv], o = sm.word_off[wv];
    while (bits) {
      int bp = __ffs(bits) - 1;
      bits &= bits - 1;
      int64_t gi = base + wv * 32 + bp;
      int64_t id = (kind == kBlocks) ? gi : int64_t(sm.pool_ids[gi >> 3]) * kBlock + (gi & 7);
      if (off + o < cap) {
        out[off + o] = int32_t(id);
        // one CTA: the pool also goes straight to shared memory for the Top-K
        if (kind == kBlocks && c.cs == 1) sm.pool_ids[off + o] = int32_t(id);
      }
      ++o;
    }
  }
  cl_sync(c);     // no rank leaves while another still reads its counters
  return total;
}

// Sum of one int per thread over the CTA (uses sm.red[1]).
__device__ int64_t block_sum(SelSmem& sm, int v) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  __syncthreads();
  if (lane == 0) sm.red[1][wid] = uint32_t(v);
  __syncthreads();
  int64_t t = 0;
  for (int i = 0; i < kSelWarps; ++i) t += sm.red[1][i];
  __syncthreads();
  return t;
}

// FP4 query: quantized exactly as the scan does; per (head, group) the
// widened codes 2 qhat (signed bytes) and the scale's (M, E).
__device__ void load_query_fp4(const IdxArgs& a, SelSmem& sm, int b) {
  const int hi = a.d.idx_heads;
  if (threadIdx.x < kMaxIdxHeads * 8) {
    const int h = threadIdx.x >> 3, g = threadIdx.x & 7;
    uint4 lo = make_uint4(0, 0, 0, 0), hi4 = make_uint4(0, 0, 0, 0);
    if (h < hi) {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.idx_q) +
                                                        (int64_t(b) * hi + h) * 128 + 16 * g);
      lo = __ldg(src);
      hi4 = __ldg(src + 1);
    }
    uint32_t sc;
    const uint2 cw = fp4_quantize_group(lo, hi4, &sc);
    reinterpret_cast<uint4*>(sm.qi + h * kQiStride)[g] =
        make_uint4(e2m1x4_to_i8x4_twice(cw.x), e2m1x4_to_i8x4_twice(cw.x >> 16), e2m1x4_to_i8x4_twice(cw.y),
                   e2m1x4_to_i8x4_twice(cw.y >> 16));
    sm.qf[h * 8 + g] = factor_e4m3(sc);
  }
  if (threadIdx.x < hi) sm.w[threadIdx.x] = a.w[int64_t(b) * hi + threadIdx.x];
  if (threadIdx.x == 0) sm.fast_exact = 1;
  __syncthreads();
}

// Query factors of sequence b: for every head its values as factors, as
// integers qi over the head's lowest set bit q_elo, the flag of the exact
// int64 path and the weights; the E4M3 value table.  One warp per head.
__device__ void load_query_factors(const IdxArgs& a, SelSmem& sm, int b) {
  const int hi = a.d.idx_heads, di = a.d.idx_dim;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const bool fp8 = a.d.idx_k_dtype == CSA2_IDXK_E4M3;
  // one warp per head (its di <= 128 channels, 4 per lane: channel lane + 32 j);
  // every global load of the warp is issued before the first use, and a head's
  // reductions stay inside its warp (no block barrier between the steps)
  static_assert(kMaxIdxHeads <= kSelWarps, "a warp per indexer head");
  constexpr int kPerLane = 128 / 32;
  const int h = wid;
  const bool head = h < hi;
  float qv[kPerLane];
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) {
    const int ch = lane + 32 * j;
    const int64_t qidx = (int64_t(b) * hi + h) * di + ch;
    qv[j] = !head || ch >= di ? 0.0f
          : fp8 ? bf16_to_f32(reinterpret_cast<const uint16_t*>(a.idx_q)[qidx])
                : reinterpret_cast<const float*>(a.idx_q)[qidx];
  }
  const float wv = threadIdx.x < hi ? a.w[int64_t(b) * hi + threadIdx.x] : 0.0f;
  if (threadIdx.x >= 512 && threadIdx.x < 512 + 256) {
    const Factor f = factor_e4m3(threadIdx.x - 512);
    sm.k_lut[threadIdx.x - 512] = f.sig * (1 << (f.exp + 9));
  }
  bool fast = true;                                   // this thread's share of the AND below
  if (h < kMaxIdxHeads) {
    Factor f[kPerLane];
    int lsb = INT_MAX;                                // lowest set bit of the head's values
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
      const int ch = lane + 32 * j;
      f[j] = factor_f32(qv[j]);
      if (head && ch < di) {
        sm.qf[ch * kMaxIdxHeads + h] = f[j];
        if (f[j].sig) lsb = min(lsb, f[j].exp + __ffs(abs(f[j].sig)) - 1);
      }
    }
    const int q_elo = __reduce_min_sync(0xFFFFFFFFu, lsb);
    bool wide = false;
    unsigned long long l1 = 0;                        // sum of |qi| (each below 2^30)
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
      const int ch = lane + 32 * j;
      if (!head || ch >= di) continue;
      int32_t q = 0;
      if (f[j].sig) {
        // q = sig * 2^exp = q * 2^q_elo; sh < 0 only drops trailing zero bits
        const int sh = f[j].exp - q_elo;
        int mag = abs(f[j].sig);
        const int bits = 32 - __clz(mag) + sh;
        if (bits > 30) {
          wide = true;
        } else {
          mag = sh >= 0 ? (mag << sh) : (mag >> -sh);
          q = f[j].sig < 0 ? -mag : mag;
          l1 += (unsigned long long)mag;
        }
      }
      sm.qi[h * kQiStride + ch] = q;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, o);
    const bool any_wide = __any_sync(0xFFFFFFFFu, wide);
    // int64 room: sum_c |qi| * max|k*2^9| (448 * 512) must stay below 2^62
    const bool qf_h = head && !any_wide && fp8 && di == 128 && l1 < (1ull << 62) / 229376ull;
    if (lane == 0) {
      sm.q_elo[h] = q_elo;
      sm.q_fast[h] = qf_h ? 1 : 0;
      sm.q_l1[h] = l1;
    }
    fast = !head || qf_h;
  }
  if (threadIdx.x < hi) sm.w[threadIdx.x] = wv;
  const int all_fast = __syncthreads_and(fast ? 1 : 0);
  if (threadIdx.x == 0) sm.fast_exact = fp8 && di == 128 && all_fast;
}

// Full mode: side 0 selects the pool over the cluster, side 1 the Top-K from a
// superset of the K best blocks (or side 0 the Top-K of the pool positions
// after the pool), the positions on rank 0 alone.  Reindex mode (cluster of
// 1): Top-K of the pool positions.
template <bool kFp4>
__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(IdxArgs a, int cs, bool reindex, bool two_sides) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  const int b = blockIdx.y;
  // This kernel starts only once the scan before it (same call) has passed its
  // own wait: the work before the call is complete.  The query, the weights,
  // the lengths and the pool, which the scan does not write, are read before
  // waiting for the scan; its scores and everything else after.
  pdl_launch_dependents();
  SelCtx c;
  c.b = b;
  c.cs = cs;
  c.rank = cs > 1 ? int(cg::this_cluster().block_rank()) : 0;
  // the length (and, for Reindex, the pool) loads go out with the query's
  // loads; their checks come after the query factors
  const int32_t n_raw = __ldg(a.ctx_len + b);
  constexpr int kPoolPer = kMaxPool / kSelThreads;
  int32_t plen_raw = 0, pin_raw[kPoolPer];
#pragma unroll
  for (int j = 0; j < kPoolPer; ++j) pin_raw[j] = -1;
  if (reindex) {
    plen_raw = __ldg(a.pool_len_in + b);
#pragma unroll
    for (int j = 0; j < kPoolPer; ++j) {
      const int i = threadIdx.x + j * kSelThreads;
      if (i < a.d.pool_blocks) pin_raw[j] = __ldg(a.pool_in + int64_t(b) * a.d.pool_blocks + i);
    }
  }
  if constexpr (kFp4)
    load_query_fp4(a, sm, b);
  else
    load_query_factors(a, sm, b);
  pdl_wait();
  c.n_ctx = check_ctx(n_raw, a.d, a.page_table != nullptr, a.ws);
  const int side = int(blockIdx.z);
  c.side = side;
  const int P = a.d.pool_blocks, K = a.d.topk;
  __syncthreads();
  int64_t nb = (c.n_ctx + kBlock - 1) / kBlock;
  // Full: the Top-K positions lie in the K best blocks (a block ahead of the
  // block of a Top-K position p holds a position ahead of p), which the pool
  // holds when K <= P or the pool is every block.  Then side 1 takes the
  // Top-K from the blocks whose bounds let them be among the K best (a
  // superset of them), at the same time as side 0 selects the pool; else
  // side 0 does both in turn and side 1 has nothing to do.
  const bool split = !reindex && two_sides && (K <= P || nb <= P);
  if (!reindex && side == 1 && !split) return;
  const int64_t p_sel = min64(P, nb);
  int32_t* blocks = side == 0 ? a.pool_out + int64_t(b) * P       // the blocks' ids (ascending)
                              : reinterpret_cast<int32_t*>(a.ws + a.L.sel_blocks) + int64_t(b) * P;
  int32_t* tk = a.topk_out + int64_t(b) * K;
  ItemKind kind = reindex ? kReindexPos : kBlocks;
  bool sup = !reindex && side == 1;
  int64_t n_items = nb, k_sel = sup ? min64(K, nb) : p_sel;
  if (reindex) {
    int32_t plen = plen_raw;
    if (plen < 0 || plen > P) { if (threadIdx.x == 0) raise_err(a.ws, CSA2_DEV_POOL); plen = 0; }
#pragma unroll
    for (int j = 0; j < kPoolPer; ++j) {
      const int i = threadIdx.x + j * kSelThreads;
      int32_t blk = i < plen ? pin_raw[j] : -1;
      if (blk >= nb) { raise_err(a.ws, CSA2_DEV_POOL); blk = -1; }
      sm.pool_ids[i] = blk;
    }
    __syncthreads();
    int my = 0;
    for (int i = threadIdx.x; i < plen; i += blockDim.x) {
      int32_t blk = sm.pool_ids[i];
      if (blk >= 0) my += int(min64(kBlock, c.n_ctx - int64_t(blk) * kBlock));
    }
    n_items = int64_t(plen) * kBlock;
    k_sel = min64(K, block_sum(sm, my));
  }
  // One call site of the selection for every phase a CTA runs (the blocks,
  // then the positions), so that a later phase finds its code in the
  // instruction cache.
  for (;;) {
    const int64_t got = certified_select<kFp4>(a, sm, c, kind, n_items, k_sel, kind == kBlocks ? blocks : tk, sup);
    if (kind != kBlocks) {
      if (c.rank == 0)
        for (int i = threadIdx.x; i < K; i += blockDim.x)
          if (i >= k_sel) tk[i] = -1;
      return;
    }
    if (sup && got > P) {          // a band too wide for the superset (ties): the pool itself, as side 0 finds it
      sup = false;
      k_sel = p_sel;
      continue;
    }
    const int64_t n_blk = sup ? got : p_sel;      // blocks the Top-K positions are taken from
    if (side == 0) {
      if (c.rank == 0) {
        for (int i = threadIdx.x; i < P; i += blockDim.x)
          if (i >= p_sel) blocks[i] = -1;
        if (threadIdx.x == 0) a.pool_len_out[b] = int32_t(p_sel);
      }
      if (split) return;
    }
    cl_sync(c);                    // every rank's block ids are written (read through L2)
    if (c.cs > 1) {
      // the positions of at most P blocks fit one CTA: rank 0 takes them alone
      // (no cluster exchange); the other ranks' shared memory is not read again
      if (c.rank != 0) return;
      c.cs = 1;
      for (int i = threadIdx.x; i < kMaxPool; i += blockDim.x) sm.pool_ids[i] = i < n_blk ? __ldcg(blocks + i) : -1;
    } else {
      for (int i = threadIdx.x; i < kMaxPool; i += blockDim.x)
        if (i >= n_blk) sm.pool_ids[i] = -1;       // ids below n_blk: written by the selection
    }
    __syncthreads();
    // valid positions of the blocks (the context's last block may be partial)
    int has_last = __syncthreads_or(threadIdx.x < kMaxPool && threadIdx.x < n_blk &&
                                    (sm.pool_ids[threadIdx.x] == nb - 1 ||
                                     (threadIdx.x + 1024 < n_blk && sm.pool_ids[threadIdx.x + 1024] == nb - 1)));
    const int64_t npos = n_blk * kBlock - (has_last ? (nb * kBlock - c.n_ctx) : 0);
    kind = kPoolPos;
    sup = false;
    n_items = n_blk * kBlock;
    k_sel = min64(K, npos);
  }
}

cudaError_t launch_select(IdxArgs a, bool reindex, cudaStream_t st) {
  // one CTA per sequence while its items fit (16,384); the block selection of a
  // longer context spreads over a cluster (up to 8 x 16,384 blocks), which
  // then also takes the positions of the pool
  const int cs = reindex ? 1 : int((a.L.nb_max + kSelCapPerCta - 1) / kSelCapPerCta);
  const size_t smem = sizeof(SelSmem);
  const bool fp4 = a.d.idx_k_dtype == CSA2_IDXK_FP4;
  // Full: the two sides side by side while both fit one wave (one CTA per
  // SM); a larger batch selects the pool and then its Top-K in one CTA set
  const bool two_sides = !reindex && int64_t(cs) * a.batch * 2 <= device_sms();
  auto kern = fp4 ? select_kernel<true> : select_kernel<false>;
  static KernelAttrs done[2];
  cudaError_t e = prepare_kernel(kern, smem, false, done[fp4 ? 1 : 0]);
  if (e != cudaSuccess) return e;
  CSA2_PROFILED(st, reindex ? "select_reindex" : "select_full",
                (e = launch_pdl(kern, dim3(unsigned(cs), unsigned(a.batch), two_sides ? 2u : 1u), dim3(kSelThreads),
                                smem, st, unsigned(cs), a, cs, reindex, two_sides)));
  return e;
}

size_t select_smem_bytes() { return sizeof(SelSmem); }

}  // namespace csa2
