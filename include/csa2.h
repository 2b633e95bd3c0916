/*
 * csa2.h -- C ABI of libcsa2.so: the CSA2 attention layer (DeepSeek-V4.1) as it
 * runs under decoder-side SWA bounded replay, on one GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is DEVICE memory allocated and owned by the caller,
 *    except `const csa2_batch *b`, which is a host struct holding device
 *    pointers, and is read during the call only.  The library allocates
 *    nothing and keeps no state between calls (the one exception is the
 *    diagnostic wait bound of csa2_set_wait_limit_ns); results are written
 *    only to the output arrays named below.
 *  - Work is enqueued on `stream` (0 = legacy default stream); no entry point
 *    synchronises the host.  Calls are thread-safe.
 *  - Return value: CSA2_OK, or a status describing an argument the host could
 *    check before launching (nothing is launched then), or CSA2_ERR_CUDA if a
 *    launch failed.
 *  - Data errors the host cannot see (an index out of range, a window without
 *    stored rows, ...) never fault: the kernel skips the offending element,
 *    keeps the rest of the result well defined, and ORs a CSA2_DERR_* bit into
 *    `*d_err` (an int32 in device memory; pass NULL to ignore).  d_err is never
 *    cleared by the library.
 *
 * Storage formats
 *  - MXFP4 (index queries and keys): E2M1 codes, two per byte, element 2i in
 *    the low nibble and 2i+1 in the high nibble; one fp32 scale per 32
 *    consecutive elements.  Scales must be powers of two in [2^-23, 2^12]
 *    (the MX scale is an E8M0 power of two); others set CSA2_DERR_SCALE and
 *    are rounded to the nearest power of two.
 *  - FP8 block-32 rows (compressed KV and SWA): 512 E4M3 (OCP "FN") codes per
 *    row plus 16 fp32 scales, one per 32 channels; value = e4m3 * scale.  The
 *    dequantised values must lie inside the f16 range (|x| < 65504).
 *  - Queries are bf16 and must lie inside the f16 range; outputs are bf16.
 *
 * Citations name the page and section that define each operation:
 *  [TAIL] "SGLang 如何让 DeepSeek V4.1 Flash 的后半层只处理尾部 token"
 *         (lab.ttaoai.cn notes on decoder SWA bounded replay), sec. 2.1-2.6.
 *  [CSA2] "DeepSeek V4.1 Flash 建模" (pages.haorui.li), CSA2 card and the
 *         Hierarchical Sparse Indexer card; mixed-precision card for formats.
 *  [D0]   SGLang/Miles day-0 article (theainews.cc), sec. 1, 2, 4.2 and 5.
 */
#ifndef CSA2_H_
#define CSA2_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *csa2_stream_t; /* same object as cudaStream_t */

#if defined(__GNUC__)
#define CSA2_API __attribute__((visibility("default")))
#else
#define CSA2_API
#endif

/* status codes */
#define CSA2_OK 0
#define CSA2_ERR_INVALID_ARG 1 /* host-checked argument error; nothing launched */
#define CSA2_ERR_UNSUPPORTED 2 /* valid request this build does not implement */
#define CSA2_ERR_CUDA 3        /* a kernel launch failed */
#define CSA2_ERR_TIMEOUT 4     /* reserved (device waits report CSA2_DERR_TIMEOUT) */
#define CSA2_ERR_TOO_LARGE 5   /* the request needs more scratch than the fixed array holds */

/* data-error bits ORed into *d_err */
#define CSA2_DERR_RANGE_IDX 1     /* a selected index outside [0, n_vis) or past kv_len */
#define CSA2_DERR_RANGE_WINDOW 2  /* a window position without a stored SWA row */
#define CSA2_DERR_RANGE_CTX 4     /* n_vis(t) exceeds the request's stored entries */
#define CSA2_DERR_SCALE 8         /* an MXFP4 scale that is not an in-range power of two */
#define CSA2_DERR_LD 16           /* a score row longer than the row stride `ld` */
#define CSA2_DERR_CAPACITY 32     /* tail rows beyond the output capacity */
#define CSA2_DERR_BAD_EXTEND 64   /* an extend with E < 0 or S < E */
#define CSA2_DERR_TIMEOUT 128     /* a pipeline wait inside a kernel gave up (internal error) */
#define CSA2_DERR_RANGE_ROW 256   /* a row index past the rows of a gather source / scatter target */
#define CSA2_DERR_NONFINITE 512   /* a NaN or infinity in a group being quantised */

/* storage formats of csa2_quantize_rows */
#define CSA2_FMT_FP8_B32 1        /* E4M3 codes + fp32 scale per 32 */
#define CSA2_FMT_FP4KV 2          /* E2M1 codes + E4M3 scale per 16 */
#define CSA2_FMT_MXFP4 3          /* E2M1 codes + power-of-two fp32 scale per 32 */

/* Rows of one layer call.  Host struct; every array is device memory.
 *   q_req[Nq]   request of each query row (0 <= q_req < num_req)
 *   q_pos[Nq]   ABSOLUTE token position t of each query row
 *   kv_start[R] pool row holding the request's compressed entry 0, in both the
 *               compressed-KV pool and the index-key pool (entry j of request
 *               r is pool row kv_start[r] + j)
 *   kv_len[R]   compressed entries stored for the request
 *   swa_start[R], swa_pos0[R], swa_len[R]: the layer's SWA rows of request r
 *               hold absolute positions swa_pos0[r] .. swa_pos0[r]+swa_len[r]-1
 *               at rows swa_start[r] .. swa_start[r]+swa_len[r]-1
 *   ratio       m in {1, 2}: each compressed entry covers m consecutive tokens
 *               without overlap, so entry j is visible to position t once its
 *               last token m*j+m-1 <= t: n_vis(t) = floor((t+1)/m)
 *               ([CSA2] CSA2 card, paragraph on the compressor; [D0] sec. 1). */
typedef struct csa2_batch {
  int32_t num_q;
  int32_t num_req;
  int32_t ratio;
  int32_t reserved;
  const int32_t *q_req;
  const int64_t *q_pos;
  const int64_t *kv_start;
  const int64_t *kv_len;
  const int64_t *swa_start;
  const int64_t *swa_pos0;
  const int64_t *swa_len;
} csa2_batch;

/* Human-readable name of a status code (static storage). */
CSA2_API const char *csa2_status_string(int status);

/* Bound on every pipeline wait inside the tensor-core kernels (index score,
 * attention), in nanoseconds of the GPU's global timer, for launches issued
 * after the call from any thread; 0 restores the default of 2 s.  When a wait
 * runs out the kernel raises CSA2_DERR_TIMEOUT, stops its pipeline, waits
 * (for at most 2 s) for the tensor-core work and copies it has in flight,
 * frees its tensor memory and returns: the outputs of that launch are
 * undefined, the CUDA context stays usable and later launches are unaffected.
 * A negative test shortens the bound so that waits run out; the pages ask
 * that such failures be reported without taking the serving process down
 * ([TAIL] sec. 2.7).  Always returns CSA2_OK. */
CSA2_API int csa2_set_wait_limit_ns(uint64_t ns);

/* ---------------------------------------------------------------------------
 * a1. Decoder bounded-replay tail layout   [TAIL] sec. 2.1, 2.2, 2.5, 2.6 and
 * the formula box: T = min(window, E); kept positions [S-T, S); lower bound S-T.
 *
 * For each request r with extend length E_r = extend_len[r] and sequence length
 * S_r = seq_len[r] after the extend, the late layers keep the last
 * T_r = min(window, E_r) rows of this extend, per request (never one cut of
 * the whole batch):
 *   tail_len[r]  = T_r                                         [R]
 *   cu_tail[r]   = T_0 + ... + T_{r-1}, cu_tail[R] = total     [R+1]
 *   for k < T_r, row i = cu_tail[r] + k:
 *     src_row[i] = cu_E[r] + E_r - T_r + k   (row in the packed extend, cu_E
 *                                             = exclusive prefix sum of E)
 *     pos[i]     = S_r - T_r + k             (absolute; never renumbered)
 *     win_lo[i]  = S_r - T_r                 (absolute window lower bound)
 *     row_req[i] = r                         (optional; may be NULL)
 * Rows at or beyond `capacity` are not written (CSA2_DERR_CAPACITY); a
 * capacity of window*num_req always suffices.  E_r < 0 or S_r < E_r gives
 * T_r = 0 and CSA2_DERR_BAD_EXTEND.  num_req >= 0; window >= 1.
 * ------------------------------------------------------------------------- */
CSA2_API int csa2_tail_layout(int32_t num_req, const int32_t *extend_len,
                     const int64_t *seq_len, int32_t window, int32_t *tail_len,
                     int32_t *cu_tail, int32_t *src_row, int64_t *pos,
                     int64_t *win_lo, int32_t *row_req, int64_t capacity,
                     int32_t *d_err, csa2_stream_t stream);

/* ---------------------------------------------------------------------------
 * a2-a4, a7. Index scores   [CSA2] CSA2 and Hierarchical cards; [D0] sec. 2
 * and sec. 5, on the FP4 indexer and its TP layout: MQA-shaped, heads
 * replicated.
 *
 *   s(q, j) = sum_h w[q,h] * max(0, sum_d Qi[q,h,d] * Ki[j,d])
 *
 * q_fp4   [Nq, n_heads, head_dim/2] MXFP4 codes;  q_scale [Nq, n_heads, head_dim/32]
 * head_w  [Nq, n_heads] fp32, or NULL for all ones
 * k_fp4   [Nk, head_dim/2];  k_scale [Nk, head_dim/32]: the index-key pool
 *         (entry j of request r at row kv_start[r] + j)
 * cand_blocks == NULL (Full / Reindex over all visible entries): row q of
 *         `scores` receives columns j = 0 .. n_vis(t)-1.
 * cand_blocks != NULL (Reindex restricted to the candidate pool): [Nq,
 *         max_blocks] ascending block ids, -1 padded; row q receives slots
 *         s = 0 .. nb*block-1 (nb = leading non-negative ids), slot s scoring
 *         entry cand_blocks[q, s/block]*block + s%block, or -inf when that
 *         entry is not visible.
 * scores  [Nq, ld] fp32, row stride ld; columns past each row's length are not
 *         written.  A row longer than ld is cut at ld (CSA2_DERR_LD); n_vis
 *         past kv_len is cut at kv_len (CSA2_DERR_RANGE_CTX).
 * Supported: head_dim == 128, n_heads in {8, 16, 32, 64}, block in [1, 64],
 * max_blocks in [1, 4096]; q_fp4, k_fp4, q_scale and k_scale 16-byte
 * aligned (CSA2_ERR_UNSUPPORTED otherwise).
 * ------------------------------------------------------------------------- */
CSA2_API int csa2_index_score(const csa2_batch *b, int32_t n_heads, int32_t head_dim,
                     const uint8_t *q_fp4, const float *q_scale,
                     const float *head_w, const uint8_t *k_fp4,
                     const float *k_scale, const int32_t *cand_blocks,
                     int32_t block, int32_t max_blocks, float *scores,
                     int64_t ld, int32_t *d_err, csa2_stream_t stream);

/* ---------------------------------------------------------------------------
 * a5, a7. Top-K selection   [CSA2] Hierarchical card; [D0] sec. 2.
 *
 * Per query, the k highest scores among its visible entries (cand_blocks ==
 * NULL, row = entries 0 .. n_vis-1) or among its visible pool slots
 * (cand_blocks != NULL, same slot map as csa2_index_score), by the total order
 * (score descending, entry id ascending).  NaN and -inf are never selected.
 *   idx   [Nq, k] selected ENTRY ids (pool slots are mapped back to entries);
 *         the first count[q] are valid, in no particular order; the rest -1.
 *   count [Nq]    min(k, number of eligible entries)
 * Supported: 1 <= k <= 2048.
 * ------------------------------------------------------------------------- */
CSA2_API int csa2_topk(const csa2_batch *b, const float *scores, int64_t ld, int32_t k,
              const int32_t *cand_blocks, int32_t block, int32_t max_blocks,
              int32_t *idx, int32_t *count, int32_t *d_err,
              csa2_stream_t stream);

/* ---------------------------------------------------------------------------
 * a5, a6. Top-K plus hierarchical candidate blocks (L20-style source)
 * [CSA2] Hierarchical card (entries grouped into blocks of 8, at most 2048
 * blocks kept);
 * [D0] sec. 2 (latest block always kept; no exclusion when everything fits).
 *
 * From full-visible scores (as csa2_index_score with cand_blocks == NULL):
 *   idx/count as csa2_topk with cand_blocks == NULL;
 *   blocks  [Nq, max_blocks]: with B = ceil(n_vis/block) blocks of `block`
 *           consecutive entries and block score = max over the block's visible
 *           entries (NaN ignored): all B blocks if B <= max_blocks, else block
 *           B-1 (it holds the latest visible position) plus the max_blocks-1
 *           best of blocks 0..B-2 by (block score desc, block id asc).  The
 *           pool is a position budget: it always holds min(B, max_blocks)
 *           blocks.  Ascending, -1 padded.
 *   nblocks [Nq]
 * Supported: 1 <= k <= 2048, block in [1, 64], max_blocks in [1, 4096].
 * ------------------------------------------------------------------------- */
CSA2_API int csa2_topk_candidates(const csa2_batch *b, const float *scores, int64_t ld,
                         int32_t k, int32_t block, int32_t max_blocks,
                         int32_t *idx, int32_t *count, int32_t *blocks,
                         int32_t *nblocks, int32_t *d_err,
                         csa2_stream_t stream);

/* ---------------------------------------------------------------------------
 * a3 + a5 streamed (NEXT-4a). Index score and top-K in one pass over the keys
 * [CSA2] Hierarchical card (the block-max, candidate and Top-K data movement
 * is a cost of its own); [D0] sec. 2 and 5.
 *
 * For full-visible rows (Full and Reindex layers scoring every visible
 * entry): the same selection as csa2_index_score (cand_blocks == NULL, ld =
 * max_len) followed by csa2_topk, without writing score rows.  A sample pass
 * scores every 8th key tile of 128 keys and sets a per-query threshold; the
 * scoring pass then appends only the (entry, score) pairs at or above it to
 * a per-query list (at most 4096 pairs); the selection is exact on any list
 * that holds at least k of them (rows of at most 4096 visible entries list
 * everything).  Rows whose list misses are rescored on the CUDA cores with
 * the scoring's own arithmetic, so the result is exact either way.
 *   max_len   bound on every row's visible entries (rows longer are cut,
 *             CSA2_DERR_LD, as with ld in csa2_index_score)
 *   idx/count as csa2_topk
 *   workspace device scratch of at least csa2_index_topk_workspace(num_q,
 *             max_len) bytes, 256-byte aligned, owned by the caller; its
 *             contents on entry do not matter and are undefined after the
 *             call.  Calls sharing one workspace must not overlap.
 * Operand layouts, flags and support as csa2_index_score; 1 <= k <= 2048.
 * ------------------------------------------------------------------------- */
CSA2_API int csa2_index_topk_workspace(int32_t num_q, int64_t max_len, int64_t *bytes);
CSA2_API int csa2_index_topk(const csa2_batch *b, int32_t n_heads, int32_t head_dim,
                             const uint8_t *q_fp4, const float *q_scale,
                             const float *head_w, const uint8_t *k_fp4,
                             const float *k_scale, int64_t max_len, int32_t k,
                             int32_t *idx, int32_t *count, void *workspace,
                             int64_t workspace_bytes, int32_t *d_err,
                             csa2_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa2_index_topk without a workspace argument, for callers that cannot
 * allocate device memory: code that runs while a CUDA graph is being
 * captured, a memory pool's own set-up code, or a host runtime that forbids
 * cudaMalloc after start-up.  The pages have no counterpart to this call; it
 * runs exactly csa2_index_topk's kernels and gives the same results.
 *
 * Its scratch is one fixed array of 64 MiB inside the library (the size is
 * csa2_index_topk_static_capacity's answer), reserved on every GPU that loads
 * the library until the process exits.  A request whose scratch
 * (csa2_index_topk_workspace(num_q, max_len)) exceeds it is rejected with
 * CSA2_ERR_TOO_LARGE and nothing is launched.  The call allocates nothing
 * (no cudaMalloc, no allocating library routine).
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and keeps it; make that first call before any
 *    stream capture, since the lookup is a runtime call of its own.
 *  - Every call, from any thread or stream, uses the same array, which keeps
 *    whatever the last call left there; each call initialises what it needs
 *    (its counters and queue are cleared by its first kernel), so leftovers
 *    never change a result.  Calls that overlap on the GPU race on the array
 *    and their results are undefined: order them (one stream, or events).
 * Arguments, outputs and flags as csa2_index_topk.
 * ------------------------------------------------------------------------- */
CSA2_API int csa2_index_topk_static_capacity(int64_t *bytes);
CSA2_API int csa2_index_topk_static(const csa2_batch *b, int32_t n_heads, int32_t head_dim,
                                    const uint8_t *q_fp4, const float *q_scale,
                                    const float *head_w, const uint8_t *k_fp4,
                                    const float *k_scale, int64_t max_len, int32_t k,
                                    int32_t *idx, int32_t *count, int32_t *d_err,
                                    csa2_stream_t stream);

/* ---------------------------------------------------------------------------
 * a8-a10. Sparse + sliding-window attention under one softmax
 * [D0] sec. 1 (own 128-token window plus at most 512 selected compressed
 * positions per query); [CSA2] mixed-precision card (the 512-dim latent row is
 * both key and value); [TAIL] sec. 2.3 (window lower bound).
 *
 * For query q (request r, position t) and head h:
 *   rows = { KV row kv_start[r]+j : j in idx[q, 0:k], j >= 0 }
 *        u { SWA row of position p : lo <= p <= t },
 *   lo   = max(win_lo[q], t - window + 1, 0)     (win_lo NULL: 0)
 *   l_i  = sm_scale * <Q[q,h,:], row_i>
 *   out[q,h,:] = sum_i e^{l_i} row_i / (sum_i e^{l_i} + e^{sink[h]})
 *   lse[q,h]   = ln(sum_i e^{l_i} + e^{sink[h]})          (sink NULL: no term)
 * The union is not de-duplicated.  Reuse layers pass an earlier layer's idx:
 * entries outside [0, n_vis(t)) or past kv_len are skipped and flagged
 * (CSA2_DERR_RANGE_IDX); idx entries are expected to be distinct.  Window
 * positions without a stored SWA row are skipped (CSA2_DERR_RANGE_WINDOW).  A
 * query with no rows gets out = 0 and lse = -inf (or sink[h]).
 *   q_bf16   [Nq, n_heads, dim] bf16;   out_bf16 [Nq, n_heads, dim] bf16
 *   kv_fp8   [Nkv, dim] + kv_scale [Nkv, dim/32]: compressed KV pool
 *   swa_fp8  [Nswa, dim] + swa_scale [Nswa, dim/32]: this layer's SWA rows
 *   idx      [Nq, k] int32 or NULL (k ignored)
 *   lse      [Nq, n_heads] fp32 or NULL
 * Supported: dim == 512, n_heads in {16, 32, 64}, 0 <= k <= 2048,
 * 1 <= window <= 1024; q_bf16, kv_fp8 and swa_fp8 16-byte aligned
 * (CSA2_ERR_UNSUPPORTED otherwise).
 * ------------------------------------------------------------------------- */
CSA2_API int csa2_sparse_swa_attn(const csa2_batch *b, int32_t n_heads, int32_t dim,
                         const void *q_bf16, const uint8_t *kv_fp8,
                         const float *kv_scale, const int32_t *idx, int32_t k,
                         const uint8_t *swa_fp8, const float *swa_scale,
                         const int64_t *win_lo, int32_t window, float sm_scale,
                         const float *sink, void *out_bf16, float *lse,
                         int32_t *d_err, csa2_stream_t stream);

/* ---------------------------------------------------------------------------
 * a10 with the FP4 main-KV layout  [CSA2] mixed-precision card (main KV as
 * E2M1 data with one E4M3 scale per 16 channels and no second-level global
 * scale: 512 x (0.5 + 1/16) = 288 B per entry; SWA stays FP8).
 *
 * The same attention as csa2_sparse_swa_attn, with the selected rows read from
 * an FP4 pool:
 *   kv_fp4 [Nkv, dim/2]  E2M1 codes, element 2i in the low nibble of byte i
 *   kv_sf  [Nkv, dim/16] E4M3 (OCP "FN") scale codes, one per 16 channels
 *   row element d = e2m1(code d) * e4m3(kv_sf[d/16])
 * Window rows are FP8 block-32 as in csa2_sparse_swa_attn.  Every other
 * argument, layout, error and limit is that function's.  kv_fp4 must be
 * 8-byte aligned.
 * ------------------------------------------------------------------------- */
CSA2_API int csa2_sparse_swa_attn_fp4kv(const csa2_batch *b, int32_t n_heads, int32_t dim,
                         const void *q_bf16, const uint8_t *kv_fp4,
                         const uint8_t *kv_sf, const int32_t *idx, int32_t k,
                         const uint8_t *swa_fp8, const float *swa_scale,
                         const int64_t *win_lo, int32_t window, float sm_scale,
                         const float *sink, void *out_bf16, float *lse,
                         int32_t *d_err, csa2_stream_t stream);

/* ---------------------------------------------------------------------------
 * Encoder-side bounded replay layout   [CSA2] Encoder Bounded Replay card
 * (on a prefix hit the last 128 cached tokens are processed again before the
 * new suffix; replayed tokens only regenerate SWA KV and never overwrite the
 * cached global KV); [D0] sec. 4.1
 * and 4.3 (local attention is cut at the rebuild boundary).
 *
 * For each request r with P_r = prefix_len[r] cached tokens (global entries
 * and index keys cached, SWA state gone) and E_r = extend_len[r] new tokens,
 * Rp_r = min(window, P_r) cached tokens are processed again before the new
 * ones:
 *   replay_len[r] = Rp_r                                            [R]
 *   cu_rows[r]    = sum over r' < r of (Rp_r' + E_r'); cu_rows[R] = total
 *   for k < Rp_r + E_r, row i = cu_rows[r] + k:
 *     pos[i]     = P_r - Rp_r + k      (absolute position)
 *     win_lo[i]  = P_r - Rp_r          (window lower bound for attention)
 *     src_row[i] = -1 for k < Rp_r     (a replayed cached token; no input row)
 *                  cu_E[r] + k - Rp_r  (row in the packed new-token input)
 *     row_req[i] = r                   (optional; may be NULL)
 *   entry_range[2r], entry_range[2r+1] (optional; may be NULL) =
 *     floor(P_r / ratio), floor((P_r + E_r) / ratio): the global entries this
 *     extend completes and writes.  Entries below the first are cached and
 *     only read; with ratio 2 and P_r odd the first new entry pairs the last
 *     cached token (a replayed row) with the first new one.
 * With Rp_r = 128 every new row's 128-token window lies inside the rebuilt
 * rows, so only replayed rows see a cut window.  ratio in {1, 2}; window >= 1.
 * Rows at or beyond `capacity` are not written (CSA2_DERR_CAPACITY).  P_r < 0
 * or E_r < 0 gives no rows for r, entry range [0, 0) and CSA2_DERR_BAD_EXTEND.
 * ------------------------------------------------------------------------- */
CSA2_API int csa2_encoder_replay_layout(int32_t num_req, const int64_t *prefix_len,
                         const int32_t *extend_len, int32_t window, int32_t ratio,
                         int32_t *replay_len, int32_t *cu_rows, int32_t *src_row,
                         int64_t *pos, int64_t *win_lo, int32_t *row_req,
                         int64_t *entry_range, int64_t capacity, int32_t *d_err,
                         csa2_stream_t stream);

/* ---------------------------------------------------------------------------
 * Row cut and scatter-back   [TAIL] sec. 2.2 (entering the late layers the
 * per-row state is cut to the tail rows; the outer layout is restored after
 * them) and sec. 2.7 (the computed tail rows are scattered back into the full
 * extend layout; the other rows are not filled in and must not be read).
 *
 * Rows are `row_bytes` bytes (a multiple of 16; src and dst 16-byte aligned,
 * not overlapping).  The rows processed are i < n, with n = *count read on
 * the device (e.g. cu_tail + num_req written by csa2_tail_layout, so no host
 * sync is needed), capped at `capacity`; count == NULL means n = capacity.
 *   gather:  dst row i          = src row row_idx[i]   (the cut)
 *   scatter: dst row row_idx[i] = src row i            (the scatter-back)
 * A negative row_idx[i] skips row i (the encoder layout's replayed rows); an
 * index >= src_rows (gather) or >= dst_rows (scatter) skips it and sets
 * CSA2_DERR_RANGE_ROW.  Rows of dst that are not written keep their bytes.
 * Scatter indices are expected to be distinct (a layout's src_row is).
 * ------------------------------------------------------------------------- */
CSA2_API int csa2_rows_gather(const int32_t *count, int64_t capacity,
                         const int32_t *row_idx, const void *src, int64_t src_rows,
                         void *dst, int64_t row_bytes, int32_t *d_err,
                         csa2_stream_t stream);
CSA2_API int csa2_rows_scatter(const int32_t *count, int64_t capacity,
                         const int32_t *row_idx, const void *src, void *dst,
                         int64_t dst_rows, int64_t row_bytes, int32_t *d_err,
                         csa2_stream_t stream);

/* ---------------------------------------------------------------------------
 * NEXT-2b. Index keys projected from the compressed main KV, written as MXFP4
 * cache rows   [CSA2] CSA2 card (compressor paragraph: the index K is
 * projected from the compressed main KV); [D0] sec. 5 (projection weights in
 * BF16 with FP32 accumulation; a fused quantise/pack/cache write keeps the
 * unfused rounding).
 *
 * For i < n:  y[i, o] = sum_d x[i, d] * w[o, d]  (fp32 accumulation on the
 * tensor cores), then row dst_row[i] of (k_fp4, k_scale) <- the MXFP4 encoding
 * of y[i, :] exactly as csa2_quantize_rows(CSA2_FMT_MXFP4) encodes an fp32
 * row.  Negative dst_row entries are skipped; entries >= rows are skipped and
 * flagged (CSA2_DERR_RANGE_ROW); groups with a NaN or infinity are written as
 * zeros (CSA2_DERR_NONFINITE); scales outside [2^-23, 2^12] set
 * CSA2_DERR_SCALE.  The pages leave the pooling of a ratio-2 pair and the
 * RoPE channels undefined: x is the compressed latent row as the caller
 * forms it, and no rotation is applied.
 *   x_bf16  [n, dim_in] bf16 (16-byte aligned);  w_bf16 [dim_out, dim_in] bf16
 *   k_fp4   [rows, dim_out/2] (16-byte aligned); k_scale [rows, dim_out/32] fp32
 * Supported: dim_in == 512, dim_out == 128.
 * ------------------------------------------------------------------------- */
CSA2_API int csa2_index_k_project(int64_t n, const void *x_bf16, int32_t dim_in,
                                  const void *w_bf16, int32_t dim_out,
                                  const int64_t *dst_row, uint8_t *k_fp4, float *k_scale,
                                  int64_t rows, int32_t *d_err, csa2_stream_t stream);

/* ---------------------------------------------------------------------------
 * Quantise-and-write of cache rows   [CSA2] mixed-precision card (main KV FP8
 * block-32, or E2M1 with one E4M3 scale per 16 channels; index K MXFP4 per
 * 32); [D0] sec. 5, on fusions that keep the quantisation semantics: fusing
 * the quantise, pack and cache write must keep the intermediate rounding and
 * scaling.
 *
 * Row i of src ([n, dim] fp32, 16-byte aligned) is quantised into row
 * dst_row[i] of a cache of `rows` rows.  Per group of G channels with
 * amax = max |x|:
 *   CSA2_FMT_FP8_B32 (G = 32): s = amax / 448 in fp32 (1 if that is 0);
 *       codes [rows, dim] E4M3(x / s); scales fp32 [rows, dim/32] = s.
 *   CSA2_FMT_FP4KV   (G = 16): sc = E4M3(amax / 6), s = value(sc);
 *       codes [rows, dim/2] E2M1(x / s) (0 if s is 0); scales uint8
 *       [rows, dim/16] = sc.
 *   CSA2_FMT_MXFP4   (G = 32): s = 2^(floor(log2 amax) - 2) (1 if amax is 0);
 *       codes [rows, dim/2] E2M1(x / s); scales fp32 [rows, dim/32] = s.  A
 *       scale outside [2^-23, 2^12] sets CSA2_DERR_SCALE (the readers'
 *       range); one that underflows to 0 writes the group as zeros, scale 1.
 * x / s is an fp32 division; E4M3 / E2M1 round to nearest, ties to even,
 * saturating at 448 / 6 (a negative value rounding to zero keeps its sign).
 * E2M1 element 2i sits in the low nibble of byte i.  A group holding a NaN or
 * infinity is written as zero codes with scale 1 (FP4KV: scale code 0) and
 * sets CSA2_DERR_NONFINITE.  dst_row[i] < 0 skips row i; dst_row[i] >= rows
 * skips it and sets CSA2_DERR_RANGE_ROW.  Destination rows are expected to
 * be distinct.  dim % G == 0, dim <= 16384; codes 16-byte aligned (FP8) or
 * 8-byte aligned (E2M1).
 * The encoder-replay write protocol uses it with the layout of
 * csa2_encoder_replay_layout: SWA rows for every processed row, global
 * entries only for [entry_range[2r], entry_range[2r+1]); cached entries are
 * never named, hence never rewritten.
 * ------------------------------------------------------------------------- */
CSA2_API int csa2_quantize_rows(int32_t format, int64_t n, const float *src, int32_t dim,
                         const int64_t *dst_row, uint8_t *codes, void *scales,
                         int64_t rows, int32_t *d_err, csa2_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H_ */
