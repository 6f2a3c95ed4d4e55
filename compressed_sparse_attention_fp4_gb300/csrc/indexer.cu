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
#include <cooperative_groups.h>

#include <cmath>

#include "common.cuh"
#include "exact.cuh"
#include "kernels.cuh"

namespace cg = cooperative_groups;

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
// Certified selection.
// ===========================================================================
enum ItemKind { kBlocks = 0, kPoolPos = 1, kReindexPos = 2 };

constexpr int kSelThreads = 1024;
constexpr int kSortCap = 4096;

struct SelSmem {
  uint32_t keyU[kSelCapPerCta];
  uint32_t keyL[kSelCapPerCta];
  uint32_t band_bits[kSelCapPerCta / 32];
  uint32_t sel_bits[kSelCapPerCta / 32];
  uint32_t word_off[kSelCapPerCta / 32];
  uint32_t hist[2][2][256];
  Factor qf[kMaxIdxHeads * 128];
  float w[kMaxIdxHeads];
  double dd[kSelThreads];
  double ps[kSelThreads];
  int32_t pool_ids[kMaxPool];
  uint32_t prefU, prefL, remU, remL;
  uint32_t cnt_in, cnt_band, cnt_sel;
  uint32_t red[32];
  int32_t n_items;
};

struct SelCtx {
  int rank, cs;       // cluster rank / size (cs = 1: this CTA alone)
  int64_t n_ctx;
  int b;
};

__device__ inline void cl_sync(const SelCtx& c) {
  if (c.cs > 1) cg::this_cluster().sync(); else __syncthreads();
}

// Block-wide exclusive scan of word popcounts of `bits` (nwords <= 512);
// returns the total.  Uses sm.red.
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
  if (lane == 31) sm.red[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t s = sm.red[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += y;
    }
    sm.red[lane] = s;   // inclusive
  }
  __syncthreads();
  uint32_t base = wid ? sm.red[wid - 1] : 0;
  if (tid < nwords) sm.word_off[tid] = base + x - v;
  uint32_t total = sm.red[31];
  __syncthreads();
  return total;
}

// Scores and keys of one item.
struct ItemVal {
  float v, delta;
  bool valid;
  int64_t id;       // emitted id: block id (kBlocks) or position
};

__device__ inline ItemVal load_item(const IdxArgs& a, ItemKind kind, const SelCtx& c,
                                    const int32_t* pool_ids, int64_t item) {
  const float* ws_f = reinterpret_cast<const float*>(a.ws);
  ItemVal r;
  r.valid = false;
  r.v = 0.0f;
  r.delta = 0.0f;
  r.id = -1;
  if (kind == kBlocks) {
    int64_t nb = (c.n_ctx + kBlock - 1) / kBlock;
    if (item < nb) {
      r.valid = true;
      r.id = item;
      r.v = ws_f[(a.L.blk_scores >> 2) + int64_t(c.b) * a.L.nb_max + item];
      r.delta = ws_f[(a.L.blk_delta >> 2) + int64_t(c.b) * a.L.nb_max + item];
    }
  } else {
    int32_t blk = pool_ids[item >> 3];
    int64_t t = int64_t(blk) * kBlock + (item & 7);
    if (blk >= 0 && t < c.n_ctx) {
      r.valid = true;
      r.id = t;
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

// Radix-select the k-th largest key of keyU and of keyL over the cluster.
__device__ void radix_two(SelSmem& sm, const SelCtx& c, int n_local, uint32_t k,
                          uint32_t& muKey, uint32_t& lamKey) {
  const int tid = threadIdx.x;
  if (tid == 0) { sm.prefU = 0; sm.prefL = 0; sm.remU = k; sm.remL = k; }
  __syncthreads();
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    uint32_t* hU = sm.hist[pass & 1][0];
    uint32_t* hL = sm.hist[pass & 1][1];
    for (int i = tid; i < 512; i += blockDim.x) (i < 256 ? hU[i] : hL[i - 256]) = 0;
    __syncthreads();
    const uint32_t pU = sm.prefU, pL = sm.prefL;
    const uint32_t maskHi = pass ? (0xFFFFFFFFu << (32 - 8 * pass)) : 0u;
    for (int i = tid; i < n_local; i += blockDim.x) {
      uint32_t u = sm.keyU[i], l = sm.keyL[i];
      if ((u & maskHi) == pU) atomicAdd(&hU[(u >> shift) & 0xFF], 1u);
      if ((l & maskHi) == pL) atomicAdd(&hL[(l >> shift) & 0xFF], 1u);
    }
    cl_sync(c);
    // warp 0 resolves U, warp 1 resolves L, on the cluster-wide histogram
    const int wid = tid >> 5, lane = tid & 31;
    if (wid < 2) {
      uint32_t cnt[8];
      uint32_t tot = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        int bucket = 255 - (lane * 8 + q);       // lane 0 holds the top buckets
        uint32_t s = 0;
        for (int r = 0; r < c.cs; ++r) {
          const uint32_t* h = sm.hist[pass & 1][wid];
          if (c.cs > 1) h = cg::this_cluster().map_shared_rank(h, r);
          s += h[bucket];
        }
        cnt[q] = s;
        tot += s;
      }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      uint32_t excl = incl - tot;
      uint32_t rem = wid == 0 ? sm.remU : sm.remL;
      bool mine = excl < rem && rem <= incl;
      uint32_t ball = __ballot_sync(0xFFFFFFFFu, mine);
      if (mine) {
        uint32_t acc = excl;
        int q = 0;
        for (; q < 8; ++q) {
          if (acc + cnt[q] >= rem) break;
          acc += cnt[q];
        }
        uint32_t bucket = 255 - (lane * 8 + q);
        if (wid == 0) { sm.prefU |= bucket << shift; sm.remU = rem - acc; }
        else { sm.prefL |= bucket << shift; sm.remL = rem - acc; }
      }
      (void)ball;
    }
    __syncthreads();
  }
  // the histograms of the last passes may still be read by other ranks
  cl_sync(c);
  muKey = sm.prefU;
  lamKey = sm.prefL;
}

// Exact score of position t (fp64), or -inf if t is out of range.
__device__ void exact_positions(const IdxArgs& a, SelSmem& sm, const SelCtx& c,
                                const int64_t* pos, int npos, double* out) {
  // tasks (position, head); one thread each; heads combined afterwards.
  const int hi = a.d.idx_heads, di = a.d.idx_dim;
  const bool fp8 = a.d.idx_k_dtype == CSA2_IDXK_E4M3;
  __syncthreads();
  for (int task = threadIdx.x; task < npos * hi; task += blockDim.x) {
    int p = task / hi, h = task % hi;
    int64_t t = pos[p];
    double d = 0.0;
    if (t >= 0 && t < c.n_ctx) {
      int64_t row = kv_row(a.page_table, a.d, c.b, t, a.ws);
      if (row >= 0) {
        if (fp8) {
          const uint8_t* kr = reinterpret_cast<const uint8_t*>(a.idx_k) + row * di;
          d = exact_head_dot(sm.qf + h * di, di, [&](int ch) { return factor_e4m3(kr[ch]); });
        } else {
          const float* kr = reinterpret_cast<const float*>(a.idx_k) + row * di;
          d = exact_head_dot(sm.qf + h * di, di, [&](int ch) { return factor_f32(kr[ch]); });
        }
      }
    }
    sm.dd[task] = d;
  }
  __syncthreads();
  for (int p = threadIdx.x; p < npos; p += blockDim.x) {
    int64_t t = pos[p];
    out[p] = (t >= 0 && t < c.n_ctx) ? combine_heads(sm.dd + p * hi, sm.w, hi) : -INFINITY;
  }
  __syncthreads();
}

// Monotone 64-bit key of a double (larger value -> larger key).
__device__ inline uint64_t f64_key(double x) {
  uint64_t u = uint64_t(__double_as_longlong(x + 0.0));
  return (u >> 63) ? ~u : (u | (uint64_t(1) << 63));
}

// One certified selection of the k best among n items of `kind`, writing the
// selected ids in ascending order to out[0 .. k).  Runs on all CTAs of the
// cluster (cs > 1, items split in rank order) or on one CTA (cs == 1).
__device__ void certified_select(const IdxArgs& a, SelSmem& sm, const SelCtx& c, ItemKind kind,
                                 int64_t n_items, int64_t k, int32_t* out,
                                 double* g_exact, int32_t* g_list, uint8_t* g_pick) {
  const int tid = threadIdx.x;
  const int64_t base = int64_t(c.rank) * kSelCapPerCta;
  const int n_local = int(max64(0, min64(kSelCapPerCta, n_items - base)));
  const int nwords = (n_local + 31) / 32;
  // ---- load keys --------------------------------------------------------
  for (int i = tid; i < kSelCapPerCta / 32; i += blockDim.x) { sm.band_bits[i] = 0; sm.sel_bits[i] = 0; }
  __syncthreads();
  for (int i = tid; i < n_local; i += blockDim.x) {
    ItemVal it = load_item(a, kind, c, sm.pool_ids, base + i);
    if (it.valid) {
      float U = __fadd_ru(it.v, it.delta);
      float L = __fadd_rd(it.v, -it.delta);
      sm.keyU[i] = f32_key(U);
      sm.keyL[i] = f32_key(L);
    } else {
      sm.keyU[i] = 0;
      sm.keyL[i] = 0;
    }
  }
  __syncthreads();
  if (k >= n_items) {
    // every valid item is selected
    for (int i = tid; i < n_local; i += blockDim.x)
      if (sm.keyU[i]) atomicOr(&sm.sel_bits[i >> 5], 1u << (i & 31));
  } else {
    uint32_t muKey, lamKey;
    radix_two(sm, c, n_local, uint32_t(k), muKey, lamKey);
    if (tid == 0) { sm.cnt_in = 0; sm.cnt_band = 0; }
    __syncthreads();
    uint32_t my_in = 0, my_band = 0;
    for (int i = tid; i < n_local; i += blockDim.x) {
      uint32_t u = sm.keyU[i], l = sm.keyL[i];
      if (u == 0) continue;
      if (l > muKey) { atomicOr(&sm.sel_bits[i >> 5], 1u << (i & 31)); ++my_in; }
      else if (u >= lamKey) { atomicOr(&sm.band_bits[i >> 5], 1u << (i & 31)); ++my_band; }
    }
    atomicAdd(&sm.cnt_in, my_in);
    atomicAdd(&sm.cnt_band, my_band);
    // ---- exact scores of this CTA's band items ----------------------------
    uint32_t nband_local = scan_words(sm, sm.band_bits, nwords);
    // gather band items (ordered) in chunks and re-score them exactly
    const int hi = a.d.idx_heads;
    const int ppi = (kind == kBlocks) ? kBlock : 1;           // positions per item
    const int chunk_items = (kSelThreads / hi) / ppi;          // items per round
    __shared__ int64_t pos_buf[kSelThreads];
    __shared__ int32_t item_buf[kSelThreads];
    for (uint32_t r0 = 0; r0 < nband_local; r0 += chunk_items) {
      // list the band items with rank in [r0, r0 + chunk_items)
      for (int wv = tid; wv < nwords; wv += blockDim.x) {
        uint32_t bits = sm.band_bits[wv];
        uint32_t o = sm.word_off[wv];
        while (bits) {
          int bpos = __ffs(bits) - 1;
          bits &= bits - 1;
          if (o >= r0 && o < r0 + chunk_items) item_buf[o - r0] = wv * 32 + bpos;
          ++o;
        }
      }
      __syncthreads();
      int nit = int(min64(chunk_items, int64_t(nband_local) - r0));
      for (int p = tid; p < nit * ppi; p += blockDim.x) {
        int64_t gi = base + item_buf[p / ppi];
        int64_t t;
        if (kind == kBlocks) t = gi * kBlock + (p % ppi);
        else {
          int32_t blk = sm.pool_ids[gi >> 3];
          t = blk < 0 ? -1 : int64_t(blk) * kBlock + (gi & 7);
        }
        pos_buf[p] = t;
      }
      __syncthreads();
      exact_positions(a, sm, c, pos_buf, nit * ppi, sm.ps);
      for (int it = tid; it < nit; it += blockDim.x) {
        double m = -INFINITY;
        for (int p = 0; p < ppi; ++p) m = fmax(m, sm.ps[it * ppi + p]);
        g_exact[base + item_buf[it]] = m;
        g_pick[base + item_buf[it]] = 0;
      }
      __syncthreads();
    }
    // ---- cluster totals ----------------------------------------------------
    cl_sync(c);
    uint32_t tot_in = 0, tot_band = 0, band_off = 0;
    for (int r = 0; r < c.cs; ++r) {
      const uint32_t* ci = &sm.cnt_in;
      const uint32_t* cb = &sm.cnt_band;
      if (c.cs > 1) { ci = cg::this_cluster().map_shared_rank(ci, r); cb = cg::this_cluster().map_shared_rank(cb, r); }
      tot_in += *ci;
      if (r < c.rank) band_off += *cb;
      tot_band += *cb;
    }
    // publish this CTA's band list (ordered) at its offset
    for (int wv = tid; wv < nwords; wv += blockDim.x) {
      uint32_t bits = sm.band_bits[wv];
      uint32_t o = sm.word_off[wv];
      while (bits) {
        int bpos = __ffs(bits) - 1;
        bits &= bits - 1;
        g_list[band_off + o] = int32_t(base + wv * 32 + bpos);
        ++o;
      }
    }
    cl_sync(c);
    // ---- rank 0 picks the best (k - tot_in) band items ----------------------
    int64_t need = k - int64_t(tot_in);
    if (c.rank == 0 && need > 0) {
      if (need >= int64_t(tot_band)) {
        for (uint32_t i = tid; i < tot_band; i += blockDim.x) g_pick[g_list[i]] = 1;
      } else if (tot_band <= kSortCap) {
        // bitonic sort of (exact key desc, item asc) in the key arrays
        uint64_t* skey = reinterpret_cast<uint64_t*>(sm.keyU);    // 4096 x 8 B
        int32_t* sidx = reinterpret_cast<int32_t*>(sm.keyL);      // 4096 x 4 B
        __syncthreads();
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
                // "before" = larger key, then smaller index
                bool i_before_j = skey[i] > skey[j] || (skey[i] == skey[j] && sidx[i] < sidx[j]);
                if (desc != i_before_j) {
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
        // large band: 64-bit radix select of the need-th largest exact score,
        // streamed over the global list by this CTA alone.
        __shared__ unsigned long long pref64;
        __shared__ uint32_t rem64, h64[256];
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
        // all keys > kappa are in; of the keys == kappa take the first rem64 by index
        uint64_t kappa = pref64;
        uint32_t take_eq = rem64;
        if (tid == 0) {
          uint32_t taken = 0;
          for (uint32_t i = 0; i < tot_band; ++i) {
            uint64_t key = f64_key(g_exact[g_list[i]]);
            if (key > kappa) g_pick[g_list[i]] = 1;
            else if (key == kappa && taken < take_eq) { g_pick[g_list[i]] = 1; ++taken; }
          }
        }
      }
    }
    cl_sync(c);
    // ---- merge picks into the selection ----------------------------------
    for (int wv = tid; wv < nwords; wv += blockDim.x) {
      uint32_t bits = sm.band_bits[wv];
      while (bits) {
        int bpos = __ffs(bits) - 1;
        bits &= bits - 1;
        if (g_pick[base + wv * 32 + bpos]) sm.sel_bits[wv] |= 1u << bpos;
      }
    }
  }
  // ---- ordered output -------------------------------------------------------
  uint32_t nsel_local = scan_words(sm, sm.sel_bits, nwords);
  if (tid == 0) sm.cnt_sel = nsel_local;
  cl_sync(c);
  uint32_t off = 0;
  for (int r = 0; r < c.rank; ++r) {
    const uint32_t* cs_ = &sm.cnt_sel;
    if (c.cs > 1) cs_ = cg::this_cluster().map_shared_rank(cs_, r);
    off += *cs_;
  }
  for (int wv = tid; wv < nwords; wv += blockDim.x) {
    uint32_t bits = sm.sel_bits[wv];
    uint32_t o = sm.word_off[wv];
    while (bits) {
      int bpos = __ffs(bits) - 1;
      bits &= bits - 1;
      int64_t gi = base + wv * 32 + bpos;
      int64_t id;
      if (kind == kBlocks) id = gi;
      else id = int64_t(sm.pool_ids[gi >> 3]) * kBlock + (gi & 7);
      if (off + o < k) out[off + o] = int32_t(id);
      ++o;
    }
  }
  // nobody may leave while another rank still reads this CTA's counters
  cl_sync(c);
}

__device__ void load_query_factors(const IdxArgs& a, SelSmem& sm, int b) {
  const int hi = a.d.idx_heads, di = a.d.idx_dim;
  const bool fp8 = a.d.idx_k_dtype == CSA2_IDXK_E4M3;
  for (int i = threadIdx.x; i < hi * di; i += blockDim.x) {
    int64_t qi = int64_t(b) * hi * di + i;
    float v = fp8 ? bf16_to_f32(reinterpret_cast<const uint16_t*>(a.idx_q)[qi])
                  : reinterpret_cast<const float*>(a.idx_q)[qi];
    sm.qf[i] = factor_f32(v);
  }
  if (threadIdx.x < hi) sm.w[threadIdx.x] = a.w[int64_t(b) * hi + threadIdx.x];
}

// Full mode: pool (cluster of cs CTAs per sequence), then Top-K over the pool
// positions (rank 0 alone).  Reindex mode (cs == 1): Top-K over pool positions.
__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(IdxArgs a, int cs, bool reindex) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  const int b = blockIdx.y;
  SelCtx c;
  c.b = b;
  c.cs = cs;
  c.rank = cs > 1 ? int(cg::this_cluster().block_rank()) : 0;
  const bool paged = a.page_table != nullptr;
  c.n_ctx = checked_ctx(a.ctx_len, a.d, b, paged, a.ws);
  load_query_factors(a, sm, b);
  const int64_t scap = a.L.sel_cap;
  double* g_exact = reinterpret_cast<double*>(a.ws + a.L.sel_exact) + int64_t(b) * scap;
  int32_t* g_list = reinterpret_cast<int32_t*>(a.ws + a.L.sel_list) + int64_t(b) * scap;
  uint8_t* g_pick = a.ws + a.L.sel_pick + int64_t(b) * scap;
  const int P = a.d.pool_blocks, K = a.d.topk;
  __syncthreads();
  if (!reindex) {
    int64_t nb = (c.n_ctx + kBlock - 1) / kBlock;
    int64_t p_sel = min64(P, nb);
    int32_t* pool = a.pool_out + int64_t(b) * P;
    certified_select(a, sm, c, kBlocks, nb, p_sel, pool, g_exact, g_list, g_pick);
    if (c.rank != 0) return;
    for (int i = threadIdx.x; i < P; i += blockDim.x) {
      if (i >= p_sel) pool[i] = -1;
    }
    if (threadIdx.x == 0) a.pool_len_out[b] = int32_t(p_sel);
    __threadfence_block();
    __syncthreads();
    for (int i = threadIdx.x; i < kMaxPool; i += blockDim.x) sm.pool_ids[i] = i < p_sel ? pool[i] : -1;
    __syncthreads();
    SelCtx c1 = c;
    c1.cs = 1;
    c1.rank = 0;
    int64_t npos = 0;
    {
      // valid pool positions (the last block of the context may be partial)
      int64_t last_blk = nb - 1;
      bool has_last = false;
      for (int i = 0; i < p_sel; ++i) has_last |= (sm.pool_ids[i] == last_blk);
      npos = p_sel * kBlock - (has_last ? (nb * kBlock - c.n_ctx) : 0);
    }
    int64_t k_sel = min64(K, npos);
    int32_t* tk = a.topk_out + int64_t(b) * K;
    certified_select(a, sm, c1, kPoolPos, p_sel * kBlock, k_sel, tk, g_exact, g_list, g_pick);
    for (int i = threadIdx.x; i < K; i += blockDim.x)
      if (i >= k_sel) tk[i] = -1;
  } else {
    int32_t plen = a.pool_len_in[b];
    if (plen < 0 || plen > P) { raise_err(a.ws, CSA2_DEV_POOL); plen = 0; }
    int64_t nb = (c.n_ctx + kBlock - 1) / kBlock;
    int64_t npos = 0;
    for (int i = threadIdx.x; i < kMaxPool; i += blockDim.x) {
      int32_t blk = i < plen ? a.pool_in[int64_t(b) * P + i] : -1;
      if (blk >= nb) { raise_err(a.ws, CSA2_DEV_POOL); blk = -1; }
      sm.pool_ids[i] = blk;
    }
    __syncthreads();
    for (int i = 0; i < plen; ++i) {
      int32_t blk = sm.pool_ids[i];
      if (blk >= 0) npos += min64(kBlock, c.n_ctx - int64_t(blk) * kBlock);
    }
    int64_t k_sel = min64(K, npos);
    int32_t* tk = a.topk_out + int64_t(b) * K;
    certified_select(a, sm, c, kReindexPos, int64_t(plen) * kBlock, k_sel, tk, g_exact, g_list, g_pick);
    for (int i = threadIdx.x; i < K; i += blockDim.x)
      if (i >= k_sel) tk[i] = -1;
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

size_t select_smem_bytes() { return sizeof(SelSmem); }

cudaError_t launch_full(IdxArgs a, cudaStream_t st) {
  const bool fp8 = a.d.idx_k_dtype == CSA2_IDXK_E4M3;
  a.err_coef = cc_err_coef(a.d.idx_dim, a.d.idx_heads);
  dim3 grid(unsigned((a.d.max_ctx + 255) / 256), unsigned(a.batch));
  if (fp8) scan_cc_kernel<true, 128><<<grid, 256, 0, st>>>(a, false);
  else scan_cc_kernel<false, 64><<<grid, 256, 0, st>>>(a, false);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  int cs = int((a.L.nb_max + kSelCapPerCta - 1) / kSelCapPerCta);
  size_t smem = sizeof(SelSmem);
  e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(cs), unsigned(a.batch), 1);
  cfg.blockDim = dim3(kSelThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, select_kernel, a, cs, false);
}

cudaError_t launch_reindex(IdxArgs a, cudaStream_t st) {
  const bool fp8 = a.d.idx_k_dtype == CSA2_IDXK_E4M3;
  a.err_coef = cc_err_coef(a.d.idx_dim, a.d.idx_heads);
  int64_t P8 = int64_t(a.d.pool_blocks) * kBlock;
  dim3 grid(unsigned((P8 + 255) / 256), unsigned(a.batch));
  if (fp8) scan_cc_kernel<true, 128><<<grid, 256, 0, st>>>(a, true);
  else scan_cc_kernel<false, 64><<<grid, 256, 0, st>>>(a, true);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  size_t smem = sizeof(SelSmem);
  e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  select_kernel<<<dim3(1, unsigned(a.batch)), kSelThreads, smem, st>>>(a, 1, true);
  return cudaGetLastError();
}

}  // namespace csa2
