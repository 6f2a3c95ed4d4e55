// common.cuh -- shared device helpers of the CSA2 decode library (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/csa2.h"

namespace csa2 {

constexpr int kLatent = CSA2_LATENT;
constexpr int kRope = CSA2_ROPE;
constexpr int kDqk = CSA2_DQK;
constexpr int kPage = CSA2_PAGE;
constexpr int kBlock = CSA2_BLOCK;
constexpr int kCodesPerRow = kLatent / 2;      // 256 bytes of E2M1 nibbles
constexpr int kScalesPerRow = kLatent / 16;    // 32 E4M3 scales
constexpr int kMaxPool = 2048;
constexpr int kMaxTopk = 2048;
constexpr int kMaxHeads = 64;
constexpr int kMaxSwa = 128;
constexpr int kMaxIdxHeads = 16;
constexpr int64_t kMaxCtx = int64_t(1) << 20;   // 8 selection CTAs x 16384 blocks
constexpr int kSelCapPerCta = 16384;           // items a selection CTA holds
constexpr int kAttnChunk = 128;                // entries per split-KV partial
constexpr int kMaxClusterSplits = 8;           // chunks merged inside one cluster (portable size)

// ---------------------------------------------------------------------------
// Workspace layout.  Computed identically on the host (sizing, validation)
// and on the device (kernels get the base pointer and this struct by value).
// ---------------------------------------------------------------------------
struct WsLayout {
  int64_t err;          // int32 error word (+ spare) -- first 256 bytes
  int64_t pos_scores;   // f32 [B][max_ctx]       Full: approximate s_t
  int64_t blk_scores;   // f32 [B][NBmax]         Full: approximate block max
  int64_t blk_delta;    // f32 [B][NBmax]         Full: error bound per block
  int64_t ri_scores;    // f32 [B][P*8]           Reindex: approx pool scores
  int64_t ri_delta;     // f32 [B][P]             Reindex: bound per pool block
  int64_t attn_o;       // f32 [B][S][H][512]     split-KV partial outputs
  int64_t attn_ml;      // f32 [B][S][H][2]       partial (max, sum)
  int64_t sel_exact;    // f64 [B][2][sel_cap]    exact scores of band items (per selection side)
  int64_t sel_list;     // i32 [B][2][sel_cap]    band item lists
  int64_t sel_pick;     // u8  [B][2][sel_cap]    band items picked
  int64_t sel_blocks;   // i32 [B][P]             Full, Top-K side: the blocks its positions come from
  int64_t total;
  int64_t nb_max;       // ceil(max_ctx / 8)
  int64_t sel_cap;      // max(NBmax, P*8): items of one selection
  int32_t splits;       // S
};

__host__ __device__ inline int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ inline int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

__host__ __device__ inline int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

// Split-KV chunks of 128 entries of an attention call: ceil((K + W) / 128),
// at least 1 (the partial path: one CTA per chunk, partials in the
// workspace's attn_o / attn_ml, merged by a combine kernel).
__host__ __device__ inline int attn_splits(const csa2_dims& d) {
  const int s = (d.topk + d.swa + kAttnChunk - 1) / kAttnChunk;
  return s < 1 ? 1 : s;
}

// Chunk c of S (cluster path) holds Top-K slots [K c / S, K (c + 1) / S) and
// then window rows up to its 128 entries, the window filled into the chunks
// in order: chunk c takes min(128 - (its Top-K slots), rows left).  With
// S = ceil((K + W) / 128) every window row finds a place.
__host__ __device__ inline int attn_chunk_main_lo(int K, int c, int S) { return int(int64_t(K) * c / S); }
__host__ __device__ inline void attn_chunk_window(int K, int W, int c, int S, int& w0, int& nw) {
  w0 = 0;
  nw = 0;
  for (int i = 0; i <= c; ++i) {
    const int room = kAttnChunk - (attn_chunk_main_lo(K, i + 1, S) - attn_chunk_main_lo(K, i, S));
    w0 += nw;
    nw = W - w0 < room ? W - w0 : room;
  }
}

// Calls with K + W <= 1024 (at most kMaxClusterSplits chunks of 128) merge
// inside thread-block clusters and use no scratch but the error word.
__host__ __device__ inline bool attn_uses_partials(const csa2_dims& d) { return attn_splits(d) > kMaxClusterSplits; }

__host__ __device__ inline WsLayout make_layout(const csa2_dims& d, int batch) {
  WsLayout L;
  int64_t off = 0;
  L.err = off; off += 256;
  L.nb_max = (d.max_ctx + kBlock - 1) / kBlock;
  L.pos_scores = off; off = align256(off + int64_t(batch) * d.max_ctx * 4);
  L.blk_scores = off; off = align256(off + int64_t(batch) * L.nb_max * 4);
  L.blk_delta = off;  off = align256(off + int64_t(batch) * L.nb_max * 4);
  int64_t pool = d.pool_blocks;
  L.ri_scores = off;  off = align256(off + int64_t(batch) * pool * kBlock * 4);
  L.ri_delta = off;   off = align256(off + int64_t(batch) * pool * 4);
  L.splits = attn_splits(d);
  L.attn_o = off;  off = align256(off + int64_t(batch) * L.splits * d.heads * kLatent * 4);
  L.attn_ml = off; off = align256(off + int64_t(batch) * L.splits * d.heads * 2 * 4);
  L.sel_cap = L.nb_max > pool * kBlock ? L.nb_max : pool * kBlock;
  L.sel_exact = off; off = align256(off + int64_t(batch) * 2 * L.sel_cap * 8);
  L.sel_list = off;  off = align256(off + int64_t(batch) * 2 * L.sel_cap * 4);
  L.sel_pick = off;  off = align256(off + int64_t(batch) * 2 * L.sel_cap);
  L.sel_blocks = off; off = align256(off + int64_t(batch) * pool * 4);
  L.total = off;
  return L;
}

// ---------------------------------------------------------------------------
// Device error word
// ---------------------------------------------------------------------------
__device__ inline void raise_err(uint8_t* ws, int bits) {
  atomicOr(reinterpret_cast<int*>(ws), bits);
}

// Physical cache row of logical position t of sequence b (-1 if the page id
// is out of range; the error bit is set by the caller's check).
__device__ inline int64_t kv_row(const int32_t* __restrict__ page_table, const csa2_dims& d,
                                 int b, int64_t t, uint8_t* ws) {
  if (page_table == nullptr) return int64_t(b) * d.max_ctx + t;
  int32_t pg = __ldg(page_table + int64_t(b) * d.max_pages + (t >> 6));
  if (pg < 0 || pg >= d.num_pages) {
    raise_err(ws, CSA2_DEV_PAGE_ID);
    return -1;
  }
  return int64_t(pg) * kPage + (t & (kPage - 1));
}

// Context length of sequence b, checked against the capacity (max_ctx, and
// max_pages * 64 for a paged cache).  A bad length is reported and treated as 0.
__device__ inline int64_t check_ctx(int64_t n, const csa2_dims& d, bool paged, uint8_t* ws) {
  if (n < 0 || n > d.max_ctx || (paged && n > int64_t(d.max_pages) * kPage)) {
    raise_err(ws, CSA2_DEV_CTX_LEN);
    return 0;
  }
  return n;
}

__device__ inline int64_t checked_ctx(const int32_t* __restrict__ ctx_len, const csa2_dims& d,
                                      int b, bool paged, uint8_t* ws) {
  return check_ctx(__ldg(ctx_len + b), d, paged, ws);
}

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------
__device__ inline float bf16_to_f32(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

// Exact value of an E4M3 byte (finite codes) as fp32.
__device__ inline float e4m3_to_f32(uint32_t c) {
  uint16_t pair = uint16_t(c & 0xFF);
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
  __half lo = __ushort_as_half(uint16_t(h2 & 0xFFFF));
  return __half2float(lo);
}

// Two E4M3 bytes (low byte = first) -> f16x2 (low half = first), exact.
__device__ inline uint32_t e4m3x2_to_f16x2(uint16_t pair) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
  return h2;
}

// Order-preserving map of a float onto uint32 (-0 is first made +0).
// Programmatic dependent launch.  The library launches its kernels with
// programmatic stream serialisation: a kernel may begin while the kernel
// before it on the stream still runs.  pdl_wait() returns once that kernel
// has completed and its writes are visible; nothing before it may read or
// write memory that other work on the stream touches.  pdl_launch_dependents()
// lets the next kernel begin its own set-up early.
__device__ inline void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ inline void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ inline uint32_t f32_key(float x) {
  uint32_t u = __float_as_uint(x + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace csa2
