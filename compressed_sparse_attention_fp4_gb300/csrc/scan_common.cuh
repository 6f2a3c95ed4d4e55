// scan_common.cuh -- pieces shared by the tensor-core indexer scans (E4M3
// keys in scan.cu, FP4 keys in scan_fp4.cu): the tile walk over the
// sequences, the key producer (a TMA ring for Full tiles, a gather of 8-row
// pool blocks for Reindex tiles), bounded waits and the tensor map.
//
// Scores (foosynaptic atlas "DeepSeek-V4.1-Flash 梗概", section 3.2,
// "Hierarchical Sparse Indexer (decoder)"): s_t = sum_h w_h ReLU(q_h . k_t)
// for every visible position (Full) or every pool position (Reindex); each
// scan writes approximate scores v_t and a rigorous per-block bound delta_j
// >= |s_t - v_t| into the workspace for the certified selection.
//
// A scan kernel's shared-memory struct provides seq_items[kSeqCache],
// n_seq_cached and abort_flag.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace csa2 {

constexpr int kTile = 128;                 // positions per tile (= MMA M)
constexpr int kGroupThreads = 128;         // threads of a query / converter / epilogue group
constexpr int kSeqCache = 64;              // sequences whose item counts sit in shared memory

__device__ inline void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(uint32_t(accumulate))
      : "memory");
}

// kind::f8f6f4 with E4M3 A and B (format code 0), fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

struct TileRef {
  int b;
  int64_t t0;        // first item
  int nvalid;        // valid items in the tile
};

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

// Warp 0: every sequence's items are read once (the first kSeqCache kept for
// the tile walks of all roles); returns the total tile count on lane 0.
template <class Sm>
__device__ inline int64_t count_tiles(const IdxArgs& a, Sm& sm, bool reindex, int lane) {
  const int ncache = min(a.batch, kSeqCache);
  int64_t tsum = 0;
  for (int b = lane; b < a.batch; b += 32) {
    const int64_t n = scan_items(a, b, reindex);
    if (b < ncache) sm.seq_items[b] = n;
    tsum += (n + kTile - 1) / kTile;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) tsum += __shfl_xor_sync(0xFFFFFFFFu, tsum, o);
  if (lane == 0) sm.n_seq_cached = ncache;
  return tsum;
}

// Global tile g -> (sequence, first item); tiles of sequence b are
// ceil(items_b / 128).  Linear walk from a hint (tiles are visited in order).
template <class Sm>
__device__ inline TileRef tile_of(const IdxArgs& a, const Sm& sm, bool reindex, int64_t g, int& hint_b,
                                  int64_t& hint_base) {
  while (true) {
    const int64_t n = hint_b < sm.n_seq_cached ? sm.seq_items[hint_b] : scan_items(a, hint_b, reindex);
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

__device__ inline void group_sync(int id) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kGroupThreads) : "memory");
}

// Bounded wait that also gives up once another role has aborted.
template <class Sm>
__device__ inline bool wait_or_abort(Sm& sm, uint64_t* bar, uint32_t parity) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = tc::globaltimer_ns();
  while (true) {
    if (tc::mbar_try_wait_sleep(bar, parity, 100000u)) return true;   // sleeps until the phase (<= 0.1 ms)
    if (sm.abort_flag) return false;
    if (tc::globaltimer_ns() - t0 > 200ull * 1000 * 1000) {
      sm.abort_flag = 1;
      return false;
    }
  }
}

__device__ inline void arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

// Ring position of a role: stage and the parity of its current use, advanced
// once per tile (no 64-bit division on the single-thread paths).
template <int kN>
struct RingPos {
  int stage = 0;
  uint32_t phase = 0;
  __device__ void next() {
    if (++stage == kN) { stage = 0; phase ^= 1u; }
  }
};

// Whether row r of the tile is a position to score, and its cache row (-1
// if not).  Issued before the epilogue waits for the MMA, so that its loads
// overlap the wait.
__device__ inline int64_t row_of(const IdxArgs& a, bool reindex, const TileRef& pt, int r) {
  if (r >= pt.nvalid) return -1;
  if (!reindex) return kv_row(a.page_table, a.d, pt.b, pt.t0 + r, a.ws);
  const bool paged = a.page_table != nullptr;
  const int64_t n_ctx = checked_ctx(a.ctx_len, a.d, pt.b, paged, a.ws);
  const int64_t item = pt.t0 + r;
  const int32_t blk = __ldg(a.pool_in + int64_t(pt.b) * a.d.pool_blocks + (item >> 3));
  const int64_t t = int64_t(blk) * kBlock + (item & 7);
  if (blk < 0 || t >= n_ctx) return -1;
  return kv_row(a.page_table, a.d, pt.b, t, a.ws);
}

// ---------------------------------------------------------------------------
// Key producer.  Rows of kRowBytes; a stage holds 128 rows.  The keys are
// read once: they go through L2 as evict-first lines, so that the stream does
// not push out the scores the scan writes (which the selection reads next).
// ---------------------------------------------------------------------------
template <int kRowBytes>
__device__ inline void issue_tile_load(const IdxArgs& a, const CUtensorMap* map, uint8_t* dst, uint64_t* full,
                                       const TileRef& tr, uint64_t policy) {
  if (a.page_table == nullptr) {
    // contiguous cache: the tile is one run of 128 rows (rows past the
    // sequence are the next one's or, past the tensor, zero-filled)
    tc::mbar_expect_tx(full, kTile * kRowBytes);
    tc::tma_load_2d_hint(map, dst, 0, int32_t(int64_t(tr.b) * a.d.max_ctx + tr.t0), full, policy);
    return;
  }
  uint32_t bytes = 0;
  int32_t rows[2];
  int nbox = (tr.nvalid > 64) ? 2 : 1;
  for (int h = 0; h < nbox; ++h) {
    int64_t t = tr.t0 + 64 * h;
    int64_t row = kv_row(a.page_table, a.d, tr.b, t, a.ws);
    rows[h] = int32_t(row);
    if (row >= 0) bytes += 64 * kRowBytes;
  }
  tc::mbar_expect_tx(full, bytes);
  for (int h = 0; h < nbox; ++h)
    if (rows[h] >= 0) tc::tma_load_2d_hint(map, dst + h * 64 * kRowBytes, 0, rows[h], full, policy);
}

// Reindex tiles: the pool blocks are scattered runs of 8 rows (never across a
// page).  Block j of a tile lands at rows 8j..8j+7 (for 128-byte swizzled
// rows, an 8-row box carries the swizzle of the whole tile).
template <int kRowBytes>
__device__ inline void gather_pool_tile(const CUtensorMap* map, uint8_t* dst, uint64_t* full, int64_t row, int lane,
                                        uint64_t policy) {
  const uint32_t nblk = __popc(__ballot_sync(0xFFFFFFFFu, row >= 0));
  if (lane == 0) tc::mbar_expect_tx(full, nblk * uint32_t(kBlock * kRowBytes));
  __syncwarp();
  if (row >= 0) tc::tma_load_2d_hint(map, dst + lane * (kBlock * kRowBytes), 0, int32_t(row), full, policy);
}

// Producer warp for Reindex tiles: resolves the cache rows of the blocks of a
// window of up to kStages tiles (pool ids and lengths, then page table: the
// loads of all its blocks in flight together), then gathers each tile with
// one 8-row TMA box per block into stage `base + stage * stride`.
// wait_first: the producer has not waited for the previous kernel yet (the
// call's inputs allowed it); it does so once the first ring of loads is out.
template <int kRowBytes, int kStages, class Sm>
__device__ inline void produce_reindex(const IdxArgs& a, const CUtensorMap* map, Sm& sm, uint8_t* base,
                                       uint32_t stride, uint64_t* full, uint64_t* empty, int64_t g0, int ntiles,
                                       int lane, bool wait_first) {
  constexpr int kResolvePer = kStages * 16 / 32;   // blocks a producer lane resolves per window
  static_assert(kResolvePer * 32 == kStages * 16, "whole windows of tiles");
  const uint64_t policy = tc::l2_policy_evict_first();
  int hb = 0;
  int64_t hbase = 0;
  bool stop = false;
  const bool paged = a.page_table != nullptr;
  RingPos<kStages> ring;
  int k = 0;
  for (int k0 = 0; k0 < ntiles && !stop; k0 += kStages) {
    const int nwin = min(kStages, ntiles - k0);
    // block idx = lane + 32 j of the window: tile idx / 16, block idx % 16
    int32_t blk[kResolvePer], pg[kResolvePer];
    int32_t nraw[kResolvePer], bq[kResolvePer];
#pragma unroll
    for (int j = 0; j < kResolvePer; ++j) {
      const int idx = lane + 32 * j;
      blk[j] = -1;
      nraw[j] = 0;
      bq[j] = 0;
      if (idx < nwin * 16) {
        const TileRef tr = tile_of(a, sm, true, g0 + k0 + idx / 16, hb, hbase);
        if ((idx % 16) * kBlock < tr.nvalid) {
          bq[j] = tr.b;
          blk[j] = __ldg(a.pool_in + int64_t(tr.b) * a.d.pool_blocks + (tr.t0 >> 3) + idx % 16);
          nraw[j] = __ldg(a.ctx_len + tr.b);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kResolvePer; ++j) {
      pg[j] = -1;
      if (blk[j] >= 0) {
        const int64_t n = check_ctx(nraw[j], a.d, paged, a.ws);
        if (int64_t(blk[j]) * kBlock >= n) blk[j] = -1;
        else if (paged) pg[j] = __ldg(a.page_table + int64_t(bq[j]) * a.d.max_pages + ((int64_t(blk[j]) * kBlock) >> 6));
      }
    }
    int64_t row[kResolvePer];
#pragma unroll
    for (int j = 0; j < kResolvePer; ++j) {
      row[j] = -1;
      if (blk[j] >= 0) {
        const int64_t t = int64_t(blk[j]) * kBlock;
        if (!paged) {
          row[j] = int64_t(bq[j]) * a.d.max_ctx + t;
        } else if (pg[j] < 0 || pg[j] >= a.d.num_pages) {
          raise_err(a.ws, CSA2_DEV_PAGE_ID);
        } else {
          row[j] = int64_t(pg[j]) * kPage + (t & (kPage - 1));
        }
      }
    }
    for (int w = 0; w < nwin; ++w, ++k, ring.next()) {
      // the lanes agree on the outcome (they issue the tile together)
      const bool free_ = k < kStages || wait_or_abort(sm, &empty[ring.stage], ring.phase ^ 1u);
      if (!__all_sync(0xFFFFFFFFu, free_)) {
        stop = true;
        break;
      }
      // tile w's 16 blocks are held by lanes 16 (w % 2) .. + 15 in register j = w / 2
      int64_t my = -1;
#pragma unroll
      for (int j = 0; j < kResolvePer; ++j) my = (j == (w >> 1)) ? row[j] : my;
      const int64_t rb = __shfl_sync(0xFFFFFFFFu, my, (lane & 15) + 16 * (w & 1));
      gather_pool_tile<kRowBytes>(map, base + size_t(ring.stage) * stride, &full[ring.stage], lane < 16 ? rb : -1,
                                  lane, policy);
    }
    if (wait_first) {
      pdl_wait();
      wait_first = false;
    }
  }
  if (wait_first) pdl_wait();
  // after an abort, let the copies still in flight land before the CTA exits
  if (sm.abort_flag && lane == 0)
    for (int j = max(0, k - kStages); j < k; ++j)
      tc::mbar_wait_bounded(&full[j % kStages], uint32_t((j / kStages) & 1), 20ull * 1000 * 1000);
}

// Producer thread for Full tiles: one TMA tile (or two page boxes) per stage.
template <int kRowBytes, int kStages, class Sm>
__device__ inline void produce_full(const IdxArgs& a, const CUtensorMap* map, Sm& sm, uint8_t* base, uint32_t stride,
                                    uint64_t* full, uint64_t* empty, int64_t g0, int ntiles, bool wait_first) {
  const uint64_t policy = tc::l2_policy_evict_first();
  int pb = 0;
  int64_t pbase = 0;
  int k = 0;
  RingPos<kStages> ring;
  for (; k < ntiles; ++k, ring.next()) {
    if (wait_first && k == kStages) {
      pdl_wait();
      wait_first = false;
    }
    if (k >= kStages && !wait_or_abort(sm, &empty[ring.stage], ring.phase ^ 1u)) break;
    issue_tile_load<kRowBytes>(a, map, base + size_t(ring.stage) * stride, &full[ring.stage],
                               tile_of(a, sm, false, g0 + k, pb, pbase), policy);
  }
  if (wait_first) pdl_wait();
  // after an abort, let the copies still in flight land before the CTA exits
  if (sm.abort_flag)
    for (int j = max(0, k - kStages); j < k; ++j)
      tc::mbar_wait_bounded(&full[j % kStages], uint32_t((j / kStages) & 1), 20ull * 1000 * 1000);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// Tensor map over the rows of an indexer-K plane: rows of row_bytes bytes;
// boxes of one page (paged Full), one tile (contiguous Full) or one pool
// block (Reindex).
inline cudaError_t idx_key_map(CUtensorMap* map, const IdxArgs& a, bool reindex, uint32_t row_bytes,
                               CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const bool paged = a.page_table != nullptr;
  const uint64_t rows = paged ? uint64_t(a.d.num_pages) * kPage : uint64_t(a.batch) * uint64_t(a.d.max_ctx);
  cuuint64_t gdim[2] = {row_bytes, rows};
  cuuint64_t gstride[1] = {row_bytes};
  cuuint32_t box[2] = {row_bytes, reindex ? uint32_t(kBlock) : (paged ? 64u : 128u)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a.idx_k), gdim, gstride, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Grid of a persistent scan: the tile count is known only on the device; the
// grid is sized for an upper bound and the CTAs split the actual tiles evenly.
inline int64_t scan_grid(const IdxArgs& a, bool reindex) {
  const int64_t items_ub = reindex ? int64_t(a.d.pool_blocks) * kBlock : a.d.max_ctx;
  const int64_t tiles_ub = int64_t(a.batch) * ((items_ub + kTile - 1) / kTile);
  const int64_t grid = min64(int64_t(device_sms()), tiles_ub);
  return grid < 1 ? 1 : grid;
}

}  // namespace csa2
