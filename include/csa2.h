/*
 * csa2.h -- C ABI of the CSA2 decode hot-path library (libcsa2.so) for
 * NVIDIA GB300 (sm_103a).
 *
 * The library implements the decode-time path of Compressed Sparse
 * Attention 2 as the pages describe it:
 *   - FP4 main-KV write: E2M1 values with one E4M3 scale per 16 channels
 *     (foosynaptic atlas "DeepSeek-V4.1-Flash 梗概", section 3.2, "FP4 main
 *     KV"; newsaint.id "DeepSeek-V4.1-Flash 2026: ...", section 4 and the
 *     FP4Quantizer of section 8);
 *   - the decoder's Hierarchical Sparse Indexer: a Full-mode scan of every
 *     visible position keeps the Top-2048 blocks of 8 as a candidate pool and
 *     Reindex layers score only inside the pool to take Top-512 (atlas,
 *     section 3.2, "Hierarchical Sparse Indexer (decoder)"; newsaint.id,
 *     section 3);
 *   - sparse MLA-style core attention over the selected FP4 main-KV entries
 *     plus an exact bf16 SWA window under one query, for the Full / Reindex /
 *     Reuse layer modes (atlas, section 3.2 mode table and figure "异构 KV";
 *     stamatios.com "DeepSeek-V4.1 Flash comprime cache KV para 890 bytes por
 *     token", section "CSA2: compressão em três dimensões").
 *
 * Conventions for every call
 *   - Pointers named as device pointers are caller-owned GPU memory; the
 *     library never allocates, frees or synchronises (except
 *     csa2_get_device_status, which reads back one word).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All work is enqueued on it, in order.
 *   - Argument errors are detected on the host, return a status code and
 *     launch nothing.
 *   - Violations that only the device can see (a context length above the
 *     capacity, a page id or a Top-K index out of range, an SWA length above
 *     the window) set bits in an error word inside the caller's workspace;
 *     the offending entry is skipped.  csa2_get_device_status reads it.
 *     No kernel traps or spins without a bound.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - Index sets are int32 logical positions, sorted ascending; -1 pads.
 *   - Ties in every ranking go to the lower index.
 *   - Inputs must be finite; NaN / Inf inputs give unspecified results.
 *
 * KV layout (main KV planes and indexer K), "rows" being cache slots:
 *   codes   uint8  [rows][256]   packed E2M1, channel 2j low nibble of byte j
 *   scales  uint8  [rows][32]    E4M3 scale of channels 16g..16g+15
 *   rope    bf16   [rows][64]    high-precision key part
 *   idx_k   E4M3   [rows][128], or fp32 [rows][64], or FP4 in two planes:
 *           codes uint8 [rows][64] (E2M1, channel 2j low nibble of byte j)
 *           followed by scales uint8 [rows][8] (E4M3, channels 16g..16g+15),
 *           the scales plane starting at idx_k + rows * 64, where rows =
 *           batch * max_ctx (contiguous) or num_pages * 64 (paged)
 * Logical position t of sequence b lives in row
 *   page_table == NULL : b * dims.max_ctx + t
 *   page_table != NULL : page_table[b * dims.max_pages + t / 64] * 64 + t % 64
 * with 64-position pages and page ids in [0, dims.num_pages).
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CSA2_LATENT 512      /* shared latent channels per main-KV entry   */
#define CSA2_ROPE 64         /* bf16 high-precision key channels           */
#define CSA2_DQK 576         /* key / query channels: latent + rope        */
#define CSA2_PAGE 64         /* positions per KV page                      */
#define CSA2_BLOCK 8         /* positions per indexer block                */

typedef enum {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad enum   */
  CSA2_ERR_UNSUPPORTED_SHAPE = 2,  /* dims outside what the kernels support   */
  CSA2_ERR_WORKSPACE_TOO_SMALL = 3,
  CSA2_ERR_CUDA = 4,               /* a CUDA runtime call failed               */
  CSA2_ERR_DEVICE_ASSERT = 5,      /* the device error word is non-zero        */
  CSA2_ERR_TIMEOUT = 6             /* a bounded device wait ran out            */
} csa2_status;

/* Bits of the device error word. */
#define CSA2_DEV_CTX_LEN   0x01  /* ctx_len[b] < 0 or > max_ctx              */
#define CSA2_DEV_PAGE_ID   0x02  /* page id outside [0, num_pages)           */
#define CSA2_DEV_TOPK_IDX  0x04  /* Top-K index outside [-1, ctx_len[b])     */
#define CSA2_DEV_SWA_LEN   0x08  /* swa_len[b] outside [0, dims.swa]         */
#define CSA2_DEV_POOL      0x10  /* pool id / pool_len out of range          */
#define CSA2_DEV_TIMEOUT   0x20  /* a bounded wait gave up                   */

typedef enum {
  CSA2_IDXK_E4M3 = 0,   /* indexer K E4M3 [rows][idx_dim], query bf16 */
  CSA2_IDXK_F32 = 1,    /* indexer K fp32 [rows][idx_dim], query fp32 */
  CSA2_IDXK_FP4 = 2     /* indexer K FP4 (two planes, idx_dim 128), query bf16,
                           quantized by the call to the same FP4 format; the
                           score is that of the dequantized query and keys */
} csa2_idxk_dtype;

typedef enum { CSA2_MODE_FULL = 0, CSA2_MODE_REINDEX = 1, CSA2_MODE_REUSE = 2 } csa2_mode;

/* Problem dimensions, shared by every call of a decode step. */
typedef struct {
  int32_t idx_heads;    /* indexer heads Hi, 1..16                            */
  int32_t idx_dim;      /* indexer dim Di: 128 (E4M3, FP4) or 64 (fp32)       */
  int32_t idx_k_dtype;  /* csa2_idxk_dtype                                    */
  int32_t pool_blocks;  /* candidate-pool blocks P, 1..2048 (pages: 2048)     */
  int32_t topk;         /* Top-K, 1..2048 (the pages use 512)                 */
  int32_t heads;        /* attention heads H, 1..64                           */
  int32_t swa;          /* SWA window rows W, 0..128                          */
  int32_t max_pages;    /* row stride of page_table (paged layout)            */
  int64_t num_pages;    /* number of physical pages (paged layout)            */
  int64_t max_ctx;      /* capacity per sequence in positions, 1..2^20;
                           also the row stride between sequences when
                           page_table == NULL                                 */
} csa2_dims;

/* Library version (major * 10000 + minor * 100 + patch). */
int32_t csa2_version(void);

/* Human-readable name of a status code (static string). */
const char* csa2_status_string(csa2_status st);

/* Bytes of workspace that indexer_full_topk, indexer_reindex_topk and
 * csa2_sparse_attn_decode need for `batch` sequences under `d`.  One
 * workspace can serve all three (calls on one stream run in order).  The
 * first 256 bytes hold the device error word; clear the whole workspace
 * (or call csa2_clear_device_status) once before first use.
 * Errors: CSA2_ERR_INVALID_ARG, CSA2_ERR_UNSUPPORTED_SHAPE. */
csa2_status csa2_workspace_size(const csa2_dims* d, int32_t batch, size_t* bytes);

/* FP4 main-KV write (atlas 3.2 "FP4 main KV"; newsaint.id section 8,
 * FP4Quantizer.quantize_and_pack).  For each row of x (bf16 [n][512],
 * device) and each group of 16 channels:
 *   s_code = E4M3(amax/6), round-to-nearest-even, saturating at 448;
 *   element nibble = sign bit << 3 | E2M1 magnitude code of |x|/s, rounded
 *   to nearest with ties to the even code (0 when s == 0).
 * Writes codes (uint8 [n][256], device) and scales (uint8 [n][32], device).
 * Errors: CSA2_ERR_INVALID_ARG (null pointer with n > 0, n < 0),
 *         CSA2_ERR_CUDA (launch failure). */
csa2_status fp4_kv_quantize(const uint16_t* x, int64_t n, uint8_t* codes,
                            uint8_t* scales, void* stream);

/* As fp4_kv_quantize, but row i of x is written to cache row dst_rows[i]
 * (int64 [n], device) -- the decode-time append of new tokens into a paged
 * or strided cache.  Rows with dst_rows[i] < 0 are skipped.  The caller
 * guarantees dst_rows[i] < rows of the cache planes. */
csa2_status fp4_kv_quantize_scatter(const uint16_t* x, int64_t n,
                                    const int64_t* dst_rows, uint8_t* codes,
                                    uint8_t* scales, void* stream);

/* fp4_kv_quantize_scatter with flags (0: the plain call).
 * CSA2_KV_EARLY_INPUTS: the operation enqueued just before this call on the
 * stream writes neither x nor dst_rows and reads or writes none of the
 * destination rows, so the rows may be written while it is still running;
 * the call still completes only after that operation has completed, so
 * later work on the stream sees the results of both.  In a decode step this
 * holds for the newest token's append enqueued after the Full layer's
 * indexer call (which reads no main-KV rows).  Other bits:
 * CSA2_ERR_INVALID_ARG. */
#define CSA2_KV_EARLY_INPUTS 1
csa2_status fp4_kv_quantize_scatter_ex(const uint16_t* x, int64_t n,
                                       const int64_t* dst_rows, uint8_t* codes,
                                       uint8_t* scales, int32_t flags, void* stream);

/* FP4 indexer-key write (the main-KV format of fp4_kv_quantize applied to
 * the indexer keys: foosynaptic atlas 3.2 "FP4 main KV" and the FP4-trained
 * indexer of newsaint.id section 4).  Row i of x (bf16 [n][128], device,
 * 16-byte aligned) is quantized per 16 channels exactly as fp4_kv_quantize
 * does and written to row dst_rows[i] (int64 [n], device; NULL: row i) of
 * the two-plane FP4 indexer-K buffer idx_k (device, 16-byte aligned) of
 * cache_rows rows: codes at idx_k + row * 64, scales at
 * idx_k + cache_rows * 64 + row * 8.  Rows whose destination is negative or
 * not below cache_rows are skipped.
 * Errors: CSA2_ERR_INVALID_ARG (null pointer with n > 0, n < 0,
 *         cache_rows < 0, misalignment, n > cache_rows without dst_rows),
 *         CSA2_ERR_CUDA. */
csa2_status fp4_idx_k_quantize_scatter(const uint16_t* x, int64_t n, const int64_t* dst_rows,
                                       uint8_t* idx_k, int64_t cache_rows, void* stream);

/* Inverse of fp4_kv_quantize: y (bf16 [n][512], device) = sign * E2M1 level
 * * E4M3 scale, which bf16 holds exactly (newsaint.id section 4: FP4 values
 * are dequantized just before attention).
 * Errors: CSA2_ERR_INVALID_ARG, CSA2_ERR_CUDA. */
csa2_status fp4_kv_dequantize(const uint8_t* codes, const uint8_t* scales,
                              int64_t n, uint16_t* y, void* stream);

/* Full-mode indexer (atlas 3.2 "Hierarchical Sparse Indexer (decoder)";
 * newsaint.id section 3 and the Full branch of HierarchicalSparseIndexer in
 * section 8).  For every sequence b (ctx_len[b] = N_b, device int32 [B]):
 *   s_t  = sum_h w_h * ReLU(q_h . k_t)           for every t < N_b,
 *   bs_j = max of s_t over block j = [8j, 8j+8),
 *   pool = Top-min(P, ceil(N_b/8)) blocks by (bs desc, j asc), ascending,
 *   topk = Top-min(K, |pool positions|) pool positions by (s desc, t asc),
 *          ascending, -1 padded.
 * Scores are ranked as if computed exactly: head dots are the exact sums
 * rounded once to fp64 and the head sum is fp64 in head order; the kernels
 * use fp32 / tensor-core scores with a rigorous error bound and re-score in
 * exact arithmetic every candidate the bound cannot decide.
 *   idx_k:   device, layout above (dtype per d->idx_k_dtype)
 *   idx_q:   device, bf16 (E4M3 and FP4 keys; 16-byte aligned for FP4) or
 *            fp32 [B][Hi][Di]
 *   w:       device, fp32 [B][Hi]
 *   pool_blocks_out: device int32 [B][P], ascending, -1 padded
 *   pool_len_out:    device int32 [B]
 *   topk_out:        device int32 [B][K]
 * The indexer-K cache may hold at most 2^31 - 1 rows (B * max_ctx
 * contiguous, num_pages * 64 paged): its tiles are addressed by 32-bit row
 * coordinates.  A larger cache is CSA2_ERR_UNSUPPORTED_SHAPE.
 * Errors: CSA2_ERR_INVALID_ARG, CSA2_ERR_UNSUPPORTED_SHAPE,
 *         CSA2_ERR_WORKSPACE_TOO_SMALL, CSA2_ERR_CUDA. */
csa2_status indexer_full_topk(const csa2_dims* d, int32_t batch,
                              const void* idx_k, const int32_t* page_table,
                              const int32_t* ctx_len, const void* idx_q,
                              const float* w, int32_t* pool_blocks_out,
                              int32_t* pool_len_out, int32_t* topk_out,
                              void* ws, size_t ws_bytes, void* stream);

/* Reindex mode (atlas 3.2: re-score with this layer's indexer query over
 * the latest Full layer's main KV / indexer K; newsaint.id section 8,
 * re-indexing branch: gather the pool's keys, score only those).  Scores
 * the positions of pool_blocks[b][0 .. pool_len[b]) with (idx_q, w) and
 * writes their Top-min(K, |pool positions|), ascending, -1 padded, with the
 * same exact ranking as indexer_full_topk.  Arguments as there; pool_blocks
 * (device int32 [B][P]) and pool_len (device int32 [B]) are the Full
 * layer's outputs. */
csa2_status indexer_reindex_topk(const csa2_dims* d, int32_t batch,
                                 const void* idx_k, const int32_t* page_table,
                                 const int32_t* ctx_len, const void* idx_q,
                                 const float* w, const int32_t* pool_blocks,
                                 const int32_t* pool_len, int32_t* topk_out,
                                 void* ws, size_t ws_bytes, void* stream);

/* indexer_full_topk / indexer_reindex_topk with flags (0: the plain calls).
 * CSA2_IDX_EARLY_INPUTS: idx_k, page_table and ctx_len (and, for Reindex,
 * pool_blocks and pool_len) are not written by the operation enqueued just
 * before this call on the stream (they were written by earlier work, before
 * that operation began), so the call may start reading them -- the scan
 * streams its first key tiles -- while that operation is still running.
 * idx_q, w, the outputs and the workspace are accessed only after it has
 * finished.  In a decode step this holds for a Full layer that follows an
 * attention call or the latent append (not the indexer-key write) and for a
 * Reindex layer that follows an attention call.  Other bits:
 * CSA2_ERR_INVALID_ARG. */
#define CSA2_IDX_EARLY_INPUTS 1
csa2_status indexer_full_topk_ex(const csa2_dims* d, int32_t batch, int32_t flags,
                                 const void* idx_k, const int32_t* page_table,
                                 const int32_t* ctx_len, const void* idx_q, const float* w,
                                 int32_t* pool_blocks_out, int32_t* pool_len_out,
                                 int32_t* topk_out, void* ws, size_t ws_bytes, void* stream);
csa2_status indexer_reindex_topk_ex(const csa2_dims* d, int32_t batch, int32_t flags,
                                    const void* idx_k, const int32_t* page_table,
                                    const int32_t* ctx_len, const void* idx_q, const float* w,
                                    const int32_t* pool_blocks, const int32_t* pool_len,
                                    int32_t* topk_out, void* ws, size_t ws_bytes, void* stream);

/* Sparse MLA-style decode attention, all layer modes (atlas 3.2 mode table
 * and figure "异构 KV": main Q reads the Top-K main-KV entries and the
 * exact SWA KV, merged; Reuse keeps KV and indices and changes only Q).
 * For every sequence b and head h, over E = {valid topk[b][i]} + {SWA rows
 * 0 .. swa_len[b]):
 *   key(e) = [dq(latent) ; rope] (576), value(e) = dq(latent) (512) for main
 *   entries, the SWA row (576) / its first 512 channels for SWA entries;
 *   logit = scale * q[b][h] . key(e);  out = softmax-weighted sum of values;
 *   lse = max logit + ln(sum exp(logit - max)); empty E: out 0, lse -inf.
 *   out is the sum of the parts of up to 8 chunks of 128 entries: for few
 *   (sequence, 32-head group) pairs each chunk runs on its own SM and the
 *   parts are added in the order the chunks finish, so repeated calls can
 *   differ in the last bits of out (lse does not); for many pairs one CTA
 *   accumulates the chunks in order and out is reproducible.
 *   mode: csa2_mode.  Indices are always supplied.  CSA2_MODE_REUSE (the
 *     layer keeps the KV and indices an earlier layer used) lets the call
 *     start reading topk, ctx_len, page_table and the main-KV planes
 *     (kv_codes, kv_scales, kv_rope) while the operation enqueued just before
 *     it on the stream is still running: in this mode those buffers must not
 *     be written by that operation (they were written by earlier work on the
 *     stream, before it began).  q, swa_kv, swa_len, out and lse are always
 *     accessed only after it has finished.  CSA2_MODE_FULL and
 *     CSA2_MODE_REINDEX read nothing before it has finished.
 *   q:        device bf16 [B][H][576], 16-byte aligned
 *   kv_codes, kv_scales, kv_rope: device, layout above (16-, 2- and
 *             16-byte aligned)
 *   topk:     device int32 [B][K], -1 = padding
 *   swa_kv:   device bf16 [B][W][576];  swa_len: device int32 [B]
 *   out:      device fp32 [B][H][512];  lse: device fp32 [B][H]
 * Errors: CSA2_ERR_INVALID_ARG, CSA2_ERR_UNSUPPORTED_SHAPE,
 *         CSA2_ERR_WORKSPACE_TOO_SMALL, CSA2_ERR_CUDA. */
csa2_status csa2_sparse_attn_decode(const csa2_dims* d, int32_t batch, int32_t mode,
                                    const uint16_t* q, const uint8_t* kv_codes,
                                    const uint8_t* kv_scales, const uint16_t* kv_rope,
                                    const int32_t* page_table, const int32_t* ctx_len,
                                    const int32_t* topk, const uint16_t* swa_kv,
                                    const int32_t* swa_len, float scale, float* out,
                                    float* lse, void* ws, size_t ws_bytes, void* stream);

/* Multi-query decode attention: q_len (1 .. CSA2_MAX_QLEN) consecutive new
 * tokens per sequence, e.g. the draft tokens a speculative step verifies
 * (stamatios.com "DeepSeek-V4.1 Flash comprime cache KV para 890 bytes por
 * token", DSpark paragraph: draft blocks over the SWA-128 window; foosynaptic
 * atlas, section 3 component table, DSpark row).  The q_len tokens are the
 * newest rows of each sequence's SWA window and share the layer's Top-K set:
 * query i (0-based, oldest first) of sequence b attends to the valid topk
 * entries and to SWA rows 0 .. swa_len[b] - (q_len - 1 - i) - 1 (its own row
 * and the older ones), with the rules of csa2_sparse_attn_decode otherwise.
 * q_len == 1 is exactly csa2_sparse_attn_decode.
 *   q:   device bf16 [B][q_len][H][576], 16-byte aligned
 *   out: device fp32 [B][q_len][H][512];  lse: device fp32 [B][q_len][H]
 *   other arguments as for csa2_sparse_attn_decode (one Top-K set, one SWA
 *   window and one swa_len per sequence).
 * Limit: for q_len > 1, topk + swa <= 1024 (at most 8 chunks of 128
 * entries, merged inside one thread-block cluster); larger shapes return
 * CSA2_ERR_UNSUPPORTED_SHAPE.
 * Errors: as csa2_sparse_attn_decode; q_len outside 1 .. CSA2_MAX_QLEN is
 *         CSA2_ERR_UNSUPPORTED_SHAPE. */
#define CSA2_MAX_QLEN 4
csa2_status csa2_sparse_attn_decode_mq(const csa2_dims* d, int32_t batch, int32_t q_len, int32_t mode,
                                       const uint16_t* q, const uint8_t* kv_codes,
                                       const uint8_t* kv_scales, const uint16_t* kv_rope,
                                       const int32_t* page_table, const int32_t* ctx_len,
                                       const int32_t* topk, const uint16_t* swa_kv,
                                       const int32_t* swa_len, float scale, float* out, float* lse,
                                       void* ws, size_t ws_bytes, void* stream);

/* Allocation-free variant of csa2_sparse_attn_decode.  The pages describe
 * no counterpart of this call; it exists for callers that must not allocate
 * GPU memory on their hot path -- e.g. a plugin running inside another
 * engine's execution step, or a serving loop whose memory budget is fixed
 * before it starts -- and so cannot provide the workspace the other calls
 * take.  The split-KV scratch lives instead in a fixed device array of
 * CSA2_NOALLOC_SCRATCH_BYTES inside the library, held on every GPU that
 * loads the library until the process exits.
 *   Limit: with S = ceil((topk + swa) / 128) chunks of entries, up to 8
 *   chunks are merged inside one thread-block cluster (or accumulated by one
 *   CTA) and need only the 256-byte error word (any batch).  Above 8 chunks the per-chunk partial
 *   outputs live in the array: 256 + B*S*H*2048 + B*S*H*8 bytes (each part
 *   rounded up to 256) must fit it -- up to batch 5 at Top-2048, SWA-128,
 *   64 heads; larger shapes return CSA2_ERR_WORKSPACE_TOO_SMALL and launch
 *   nothing.
 *   Arguments and results are those of csa2_sparse_attn_decode without
 *   ws / ws_bytes; err_word (device int32, may be NULL) receives the device
 *   error bits of this call, ORed in.
 *   The first call on a device looks up the array's device address (once
 *   per device, with that device current); make that first call before any
 *   stream capture.  The call allocates nothing (no cudaMalloc / cudaFree).
 *   All calls share the one array and it keeps the last call's contents:
 *   calls whose GPU work can overlap (e.g. on unsynchronised streams) race
 *   on it and must be serialised by the caller. */
#define CSA2_NOALLOC_SCRATCH_BYTES (12u << 20)
csa2_status csa2_sparse_attn_decode_noalloc(const csa2_dims* d, int32_t batch, int32_t mode,
                                            const uint16_t* q, const uint8_t* kv_codes,
                                            const uint8_t* kv_scales, const uint16_t* kv_rope,
                                            const int32_t* page_table, const int32_t* ctx_len,
                                            const int32_t* topk, const uint16_t* swa_kv,
                                            const int32_t* swa_len, float scale, float* out,
                                            float* lse, int32_t* err_word, void* stream);

/* Kernel timing, a tracing aid.  While enabled, the library brackets every
 * kernel it launches with a pair of CUDA events on the launching stream
 * (not for use during stream capture).  Enabling (or disabling) clears the
 * records.  csa2_profile_read waits for the recorded events and returns per
 * kernel name the number of launches and their summed milliseconds in
 * out[0 .. min(*n_entries, max_entries)), *n_entries = number of kernels. */
typedef struct {
  char name[32];
  int32_t launches;
  double total_ms;
} csa2_kernel_time;
csa2_status csa2_profile_enable(int32_t on);
csa2_status csa2_profile_read(csa2_kernel_time* out, int32_t max_entries, int32_t* n_entries);

/* Copies the device error word of `ws` to *word (synchronising `stream`)
 * and returns CSA2_OK if it is zero, CSA2_ERR_DEVICE_ASSERT otherwise. */
csa2_status csa2_get_device_status(const void* ws, void* stream, int32_t* word);

/* Zeroes the device error word of `ws` (enqueued on `stream`). */
csa2_status csa2_clear_device_status(void* ws, void* stream);

/* Self-test of the device timeout path.  Enqueues one small kernel whose
 * thread waits, with the bounded mbarrier wait every library kernel uses, on
 * an mbarrier that nothing arrives at; after limit_us microseconds
 * (1 .. 1,000,000) the wait gives up, CSA2_DEV_TIMEOUT is set in the error
 * word of ws (device, 256-byte aligned, ws_bytes >= 256) and the kernel
 * returns: no fault, no trap, the context stays usable.
 * Errors: CSA2_ERR_INVALID_ARG, CSA2_ERR_CUDA. */
csa2_status csa2_selftest_wait_timeout(void* ws, size_t ws_bytes, uint32_t limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H */
