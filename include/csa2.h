/*
 * csa2.h — C ABI of libcsa2.so, the B300 (sm_103a) hot path of Compressed
 * Sparse Attention 2 (CSA2) over a shared main-KV cache held in FP4.
 *
 * Page citations used below:
 *  [CSA2] wire.sakhanda.co, "DeepSeek AI выпустила DeepSeek-V4.1-Flash с
 *         контекстом в 1 млн токенов, KV-кэшем FP4 и повторным
 *         использованием внимания между слоями", section "Сжатое разреженное
 *         внимание 2 (CSA2)": layer modes Full / Reindex / Reuse, Top-512,
 *         each layer's own main Q and SWA KV, the hierarchical pool of up to
 *         2048 blocks x 8 positions formed by the Full layer.
 *  [FP4]  same page, section "FP4 KV, ограниченное повторное проигрывание и
 *         другие расширения": main KV in E2M1 with one E4M3 scale per 16
 *         channels, without NVFP4's global scale.
 *  [CED]  same page, section "Каузальный энкодер-декодер: вдвое меньший
 *         префилл": every layer keeps 128-token sliding-window attention.
 *  [TG]   tgviewer.app, "DeepSeek-V4.1-Flash: Frontier Agents on a Smaller
 *         Memory Budget", CSA2 bullet: sharing Top-K indices removes
 *         re-scoring the whole history.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates. Scratch memory comes from a caller-provided workspace
 *    of at least csa2_workspace_size(...) bytes, 256-byte aligned.
 *  - Every tensor base must be 16-byte aligned; rows are packed (no padding)
 *    unless a stride argument says otherwise. Strides are in ROWS.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and returns without synchronising the host; results are valid
 *    once the stream reaches that point. Calls are capturable in CUDA graphs
 *    (no host synchronisation, no allocation; memsets are async).
 *  - The return value is a csa2_status. Host-side validation failures
 *    return before enqueuing anything. Device-side checks (an index or a
 *    length out of range) never trap: the offending access is skipped and,
 *    when `d_status` (a device int32, caller-zeroed) is non-NULL, the first
 *    failing code is written there with an atomic compare-and-swap.
 *  - Formats: bf16 tensors are IEEE bfloat16; E4M3 tensors are raw bytes of
 *    the OCP FP8 E4M3 ("fn") format; the FP4 main-KV cache is two planes,
 *    `codes` [.., d/2] (two E2M1 codes per byte, channel 2i in the low
 *    nibble, bit 3 of a code = sign) and `scales` [.., d/16] (E4M3).
 *  - Layout symbols: B sequences (or prefill queries), n positions, d = 512
 *    main dim, H main query heads (multiple of 16, <= 64), H_I <= 8 indexer
 *    heads, d_I in {64, 128} indexer dim, k <= 2048 Top-K, W <= 128 window.
 */
#ifndef CSA2_H_
#define CSA2_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CSA2_API __attribute__((visibility("default")))
#else
#define CSA2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
enum csa2_status {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1,      /* NULL / misaligned pointer, bad value      */
  CSA2_ERR_UNSUPPORTED_SHAPE = 2,/* a size outside what the kernels support  */
  CSA2_ERR_WORKSPACE = 3,        /* workspace missing or too small           */
  CSA2_ERR_CUDA = 4,             /* a CUDA launch or memset failed           */
  CSA2_ERR_TIMEOUT = 5,          /* a bounded device wait gave up            */
  CSA2_ERR_DEVICE_BOUNDS = 6,    /* (device) an index/length was out of range */
  CSA2_ERR_DEVICE_RANGE = 7      /* (device) an input value outside the range the
                                    kernel represents exactly (see the call)  */
};

/* Human-readable name of a status code (static string, never NULL). */
CSA2_API const char* csa2_status_string(int status);

/* Name and text of the last CUDA error that made a call of the calling
 * host thread return CSA2_ERR_CUDA ("" if none; static per-thread storage,
 * valid until that thread's next failing call). */
CSA2_API const char* csa2_last_cuda_error(void);

/* Library ABI version (major*100 + minor). */
CSA2_API int csa2_version(void);

/* Number of kernel launches this process has issued through the library
 * (host-side counter; graph replays of captured launches are not counted). */
CSA2_API uint64_t csa2_launch_count(void);

/* ---- test hook: bounded device waits -------------------------------------- */
/* Every wait inside the kernels (on a tile, an accumulator, or the other CTA
 * of a pair) gives up after a bound, reports CSA2_ERR_TIMEOUT through
 * d_status, releases what the CTA holds (tensor memory) and returns; nothing
 * hangs or traps. This hook lets tests exercise that path without faulting
 * the GPU: with `fault` != CSA2_FAULT_NONE, every later launch of that kernel
 * withholds one signal (its producers never hand over their last tile), so
 * its consumers' waits run out. `wait_ns` sets the bound of every device wait
 * (0 = the default, 2 s). Process-wide; not for production use. The pages
 * have no counterpart: this exists to test the library's own failure path. */
enum csa2_fault {
  CSA2_FAULT_NONE = 0,
  CSA2_FAULT_ATTN = 1,       /* sparse attention (csa2_sparse_attn, groups)  */
  CSA2_FAULT_SCAN = 2,       /* Full indexer scan (TMA-fed form)             */
  CSA2_FAULT_PREFILL = 3     /* prefill indexer GEMM                         */
};
CSA2_API int csa2_debug_set_fault(int32_t fault, int64_t wait_ns);

/* ---- workspace sizing -------------------------------------------------- */
enum csa2_op {
  CSA2_OP_TOPK = 1,          /* csa2_topk                                  */
  CSA2_OP_INDEX_FULL = 2,    /* csa2_index_full (scores + Top-K)           */
  CSA2_OP_INDEX_REINDEX = 3, /* csa2_index_reindex                         */
  CSA2_OP_FORM_POOL = 4,     /* csa2_form_pool                             */
  CSA2_OP_SPARSE_ATTN = 5,   /* csa2_sparse_attn (split-K partials)        */
  CSA2_OP_LAYER_GROUP = 6,   /* csa2_layer_group (max of the above)        */
  CSA2_OP_PREFILL_GROUP = 7, /* csa2_prefill_group: B = queries, n_max = entries */
  CSA2_OP_FORM_POOL_BLOCK_MAX = 8 /* csa2_form_pool_block_max (n_max = positions) */
};

/* Bytes of workspace an op needs for B rows of at most n_max candidates,
 * Top-k, pool P blocks and H heads (arguments an op does not use are
 * ignored). Returns 0 for an unknown op. */
CSA2_API size_t csa2_workspace_size(int32_t op, int32_t B, int64_t n_max, int32_t k,
                           int32_t P, int32_t H);

/* ---- a1: FP4 quantise / append [FP4] ----------------------------------- */
/* Quantise bf16 main-KV rows to E2M1 codes with one E4M3 scale per 16
 * channels (no global scale) and store them in the cache. Per group of 16
 * channels: scale = E4M3(amax / 6) rounded to nearest even with saturation;
 * code_c = sign(x_c) | E2M1(|x_c| / scale) rounded to nearest even with
 * saturation at 6; a group whose scale is zero stores +0 codes. The result
 * is bit-exact (IEEE fp32 division, hardware RNE conversions).
 *   x      [B][rows][d] bf16
 *   pos    [B] int64 device (NULL = all zero): row r of sequence b goes to
 *          cache position pos[b] + r
 *   codes  [B][n_cap][d/2] u8, scales [B][n_cap][d/16] u8
 * Rows whose position is >= n_cap are skipped (CSA2_ERR_DEVICE_BOUNDS). */
CSA2_API int csa2_quantize_kv_fp4(const void* x, int32_t B, int64_t rows, int32_t d,
                         const int64_t* pos, uint8_t* codes, uint8_t* scales,
                         int64_t n_cap, int32_t* d_status, void* stream);

/* ---- a2: indexer-K append + block means [CSA2] ------------------------- */
/* Copy E4M3 indexer-key rows into the cache and refresh the mean key of
 * every aligned 8-position block they touch (the pool is formed over
 * blocks of 8 positions). A block's mean covers its positions from the
 * block start through the last appended position: the exact fp32 sum of
 * the present keys divided by their count, rounded to E4M3 (RNE, sat).
 *   k_new [B][rows][d_I] u8; pos [B] int64 device (NULL = 0)
 *   kI    [B][n_cap][d_I] u8; kbar [B][ceil(n_cap/8)][d_I] u8 */
CSA2_API int csa2_append_indexer_k(const uint8_t* k_new, int32_t B, int64_t rows,
                          int32_t d_I, const int64_t* pos, uint8_t* kI,
                          uint8_t* kbar, int64_t n_cap, int32_t* d_status,
                          void* stream);

/* Recompute every block mean of positions [0, n[b]) from an indexer-K cache
 * that was filled in place (bulk prefill). n [B] int64 device, each
 * <= n_max <= n_cap. */
CSA2_API int csa2_block_means(const uint8_t* kI, int32_t B, int32_t d_I,
                     const int64_t* n, int64_t n_max, int64_t n_cap,
                     uint8_t* kbar, int32_t* d_status, void* stream);

/* Append one bf16 sliding-window row per sequence into the layer's ring:
 * slot = pos[b] mod W [CED].
 *   x [B][d] bf16; pos [B] int64 device; swa [B][W][d] bf16 */
CSA2_API int csa2_append_swa(const void* x, int32_t B, int32_t d, const int64_t* pos,
                    void* swa, int32_t W, void* stream);

/* Sliding-window rings and token order [CED]. Each layer keeps the last W
 * tokens' rows in a ring: token t of sequence b at slot t mod W. After n[b]
 * tokens the window is tokens n - c .. n - 1, c = min(n[b], W).
 * csa2_swa_export copies every layer's window out in token order:
 * rows_out[l][b][i] = the row of token n - c + i for i < c, zero rows after.
 * csa2_swa_restore writes rows given in that order back into their slots
 * (the buffer side of restoring a session whose window rows were saved or
 * recomputed; the recomputation itself needs weights and is not here) and,
 * if swa_len_out is not NULL, sets swa_len_out[b] = c.
 *   rings, rows  HOST arrays [L] of device [B][W][d] bf16; n [B] int64 device.
 *   d = 512, L <= 64. */
CSA2_API int csa2_swa_export(const void* const* rings, int32_t L, int32_t W, int32_t B,
                             int32_t d, const int64_t* n, void* const* rows_out,
                             void* stream);
CSA2_API int csa2_swa_restore(const void* const* rows, int32_t L, int32_t W, int32_t B,
                              int32_t d, const int64_t* n, void* const* rings,
                              int32_t* swa_len_out, void* stream);

/* Append one decode token to every cache of a layer stack in ONE launch:
 * the main-KV row x_b (FP4, exactly as csa2_quantize_kv_fp4), the indexer
 * key (with its block mean, exactly as csa2_append_indexer_k; kbar may be
 * NULL) and each layer's SWA row (as csa2_append_swa), all at pos[b].
 *   kv_new [B][d] bf16; kI_new [B][d_I] u8
 *   swa_new, swa: HOST arrays of L device pointers ([B][d] bf16 new rows,
 *   [B][W][d] bf16 rings); L <= 64. Other arrays as in the calls above. */
CSA2_API int csa2_append_step(const void* kv_new, const uint8_t* kI_new,
                              const void* const* swa_new, void* const* swa,
                              int32_t L, int32_t W, int32_t B, int32_t d,
                              int32_t d_I, const int64_t* pos, uint8_t* codes,
                              uint8_t* scales, uint8_t* kI, uint8_t* kbar,
                              int64_t n_cap, int32_t* d_status, void* stream);

/* Encoder-style append at compression ratio `ratio` (tokens per compressed
 * main-KV entry; ratio 1 is csa2_append_step). pos[b] is the new token's
 * position t. Every call writes each layer's SWA row into slot t % W. The
 * compressed entry (kv_new, kI_new: an input, since merging tokens into an
 * entry needs weights) is appended, with its block mean refreshed, only
 * when it completes at this token: at entry index (t + 1) / ratio - 1 when
 * (t + 1) % ratio == 0 (checked per sequence on the device, so the launch is
 * the same every step). When not NULL, n_vis_out[b] = (t + 1) / ratio (the
 * entries the token sees) and swa_len_out[b] = min(t + 1, W) are written.
 * Arrays as in csa2_append_step. */
CSA2_API int csa2_append_step_ratio(const void* kv_new, const uint8_t* kI_new,
                                    const void* const* swa_new, void* const* swa,
                                    int32_t L, int32_t W, int32_t B, int32_t d,
                                    int32_t d_I, const int64_t* pos, int32_t ratio,
                                    uint8_t* codes, uint8_t* scales, uint8_t* kI,
                                    uint8_t* kbar, int64_t n_cap, int64_t* n_vis_out,
                                    int32_t* swa_len_out, int32_t* d_status,
                                    void* stream);

/* ---- a3: indexer scores [CSA2] ------------------------------------------ */
/* Raw indexer scan: scores[b][t] = sum_h w[b][h] * relu(qI[b][h] . kI[b][t])
 * for t < n[b], FP8 x FP8 products accumulated in fp32 on the tensor cores
 * (one indexer key per position shared by all heads; no 1/sqrt(d_I)).
 *   qI [B][H_I][d_I] u8 (E4M3); w [B][H_I] fp32
 *   kI row (b,t) at kI + (b*kI_seq_stride + t)*d_I (stride 0 = one shared cache)
 *   n [B] int64 device, every n[b] <= n_max (else CSA2_ERR_DEVICE_BOUNDS)
 *   scores [B][scores_stride] fp32 */
CSA2_API int csa2_index_scores(const uint8_t* qI, const float* w, const uint8_t* kI,
                      int64_t kI_seq_stride, const int64_t* n, int32_t B,
                      int32_t H_I, int32_t d_I, int64_t n_max, float* scores,
                      int64_t scores_stride, int32_t* d_status, void* stream);

/* ---- a6: Top-K [CSA2] --------------------------------------------------- */
/* Select, per row b, the k best of its first n[b] candidates by (score
 * descending, position ascending); write their positions sorted ascending
 * to idx_out[b][0..k), padded with -1 when fewer than k candidates exist.
 *   scores [B][scores_stride] fp32 (not NaN)
 *   cand_pos [B][scores_stride] int32 or NULL: candidate i of row b has
 *            position cand_pos[b][i] (-1 = absent); NULL means position i.
 *   n        [B] int64 device, or NULL: every row has n_max candidates.
 *   k <= 2048. Workspace: CSA2_OP_TOPK. */
CSA2_API int csa2_topk(const float* scores, const int32_t* cand_pos,
              int64_t scores_stride, const int64_t* n, int32_t B,
              int64_t n_max, int32_t k, int32_t* idx_out, void* ws,
              size_t ws_bytes, void* stream);

/* ---- Top-K without a caller workspace ----------------------------------- */
/* The source pages have no counterpart to this call; it exists for callers
 * of this library that cannot allocate device memory: code running inside
 * another runtime's execution hook where allocation is forbidden (an
 * inference-engine plugin's enqueue, say), steady-state serving loops that
 * must never call cudaMalloc because it can synchronise the whole device,
 * and plain C callers with no allocator of their own.
 * Same selection, arguments and result as csa2_topk, minus the workspace:
 * the scratch lives in a fixed device array inside the library, reserved on
 * every GPU that loads the library and held until the process exits
 * (7,341,056 bytes = 7.0 MiB, the csa2_topk workspace of
 * CSA2_TOPK_NOALLOC_MAX_ROWS rows). Limits: at most CSA2_TOPK_NOALLOC_MAX_ROWS rows (B);
 * larger B returns CSA2_ERR_UNSUPPORTED_SHAPE and enqueues nothing.
 * The first call made while a device is current looks up that device's
 * array address (one-time set-up); make that first call before capturing
 * any stream. All calls share the one array and each call re-zeroes what
 * must start at zero, so calls whose GPU work overlaps (different streams,
 * or unordered host threads) race and return wrong results: order them on
 * one stream. Calls no cudaMalloc/cudaFree or allocating routine. */
#define CSA2_TOPK_NOALLOC_MAX_ROWS 64
CSA2_API int csa2_topk_noalloc(const float* scores, const int32_t* cand_pos,
                               int64_t scores_stride, const int64_t* n,
                               int32_t B, int64_t n_max, int32_t k,
                               int32_t* idx_out, void* stream);

/* ---- a3+a6: Full layer indexer [CSA2] ----------------------------------- */
/* Full mode: score every visible position t < n[b] (csa2_index_scores) and
 * select a new Top-k (csa2_topk), with the Top-K histogram fused into the
 * scan. scores_out (NULL allowed) receives the scores [B][n_max].
 * Workspace: CSA2_OP_INDEX_FULL. */
CSA2_API int csa2_index_full(const uint8_t* qI, const float* w, const uint8_t* kI,
                    int64_t kI_seq_stride, const int64_t* n, int32_t B,
                    int32_t H_I, int32_t d_I, int64_t n_max, int32_t k,
                    int32_t* idx_out, float* scores_out, void* ws,
                    size_t ws_bytes, int32_t* d_status, void* stream);

/* ---- a4: hierarchical pool [CSA2] --------------------------------------- */
/* The Full layer forms a bounded candidate pool: every block of 8 positions
 * is scored on its mean key (kbar) with the pool-forming indexer query, and
 * the best min(P, ceil(n/8)) blocks (score desc, block id asc) are written
 * to pool_out[b][0..P) sorted ascending, -1 padded. P <= 2048.
 *   kbar row (b,j) at kbar + (b*kbar_seq_stride + j)*d_I
 * Workspace: CSA2_OP_FORM_POOL (with n_max = positions, not blocks). */
CSA2_API int csa2_form_pool(const uint8_t* qI, const float* w, const uint8_t* kbar,
                   int64_t kbar_seq_stride, const int64_t* n, int32_t B,
                   int32_t H_I, int32_t d_I, int64_t n_max, int32_t P,
                   int32_t* pool_out, void* ws, size_t ws_bytes,
                   int32_t* d_status, void* stream);

/* ---- pool by the max-of-token rule --------------------------------------- */
/* A variant of the pool with guaranteed recall. The pages give no block
 * score; this one scores block j with the largest of the Full layer's token
 * scores over its positions 8j .. 8j+7 below n[b], instead of scoring the
 * block's mean key. A block holding any of the Full Top-k positions then
 * scores at least the k-th score, so for P >= k the pool contains every one
 * of them (the mean-key rule gives no such guarantee: relu is convex).
 *   scores    [B][scores_stride] fp32 (a Full scan's output, not NaN)
 *   n, n_max  as in csa2_topk (n = positions; blocks = ceil(n/8))
 *   pool_out  [B][P] ascending block ids, -1 padded; P <= 2048
 * Workspace: CSA2_OP_FORM_POOL_BLOCK_MAX. */
CSA2_API int csa2_form_pool_block_max(const float* scores, int64_t scores_stride,
                                      const int64_t* n, int32_t B, int64_t n_max,
                                      int32_t P, int32_t* pool_out, void* ws,
                                      size_t ws_bytes, void* stream);

/* ---- a5+a6: Reindex layer [CSA2] ---------------------------------------- */
/* Reindex mode: rescore only the positions of the pool's blocks (pool
 * [B][P] ascending block ids, -1 = empty; positions >= n[b] are absent)
 * with this layer's own indexer query, then select Top-k over them.
 * Workspace: CSA2_OP_INDEX_REINDEX. */
CSA2_API int csa2_index_reindex(const uint8_t* qI, const float* w, const uint8_t* kI,
                       int64_t kI_seq_stride, const int64_t* n,
                       const int32_t* pool, int32_t P, int32_t B, int32_t H_I,
                       int32_t d_I, int32_t k, int32_t* idx_out, void* ws,
                       size_t ws_bytes, int32_t* d_status, void* stream);

/* ---- a7+a8+a9: sparse attention over FP4 rows + SWA [CSA2][CED][FP4] --- */
/* out[b][h] = softmax(scale * q[b][h] . X^T) X over the keys X = the
 * dequantised main-KV rows idx[b][0..k) (-1 = absent; main K = V) followed
 * by the present rows of the sequence's SWA window (K = V, bf16).
 * Q.K^T and P.V run on the tcgen05 tensor cores with fp16 operands and fp32
 * accumulation (TMEM). The FP4 dequantisation (E2M1 x E4M3, at most 6
 * significant bits in 2^-10 .. 2688) is exact in fp16. Each query head is
 * scaled by the power of two that brings its largest magnitude into
 * [2^14, 2^15), which makes every bf16 query exact (the factor is folded into
 * the head's softmax scale). An SWA row whose largest magnitude reaches 2^16
 * is scaled by 2^-b (b <= 7), with its logits and probabilities scaled back
 * exactly; rows reaching 2^23 saturate and set CSA2_ERR_DEVICE_RANGE. SWA
 * values below 2^-14 keep an absolute accuracy of 2^-25. Probabilities are
 * rounded to fp16 and the softmax denominator sums the rounded values; logits
 * must be finite in fp32. Key tiles beyond one CTA are split-K partials
 * merged by log-sum-exp. A row with no key at all gets zeros.
 *   q, out   [B][H][d] bf16
 *   codes/scales row (b,t) at (b*kv_seq_stride + t); t must be < n_cap
 *            (checked: CSA2_ERR_DEVICE_BOUNDS, key skipped)
 *   idx      [B][k] int32
 *   swa      the W-row SWA window of sequence b starts at row b*swa_seq_stride
 *            (decode rings: stride W; a prefill chunk: stride 1, the array
 *            holding the rows of tokens p0-W+1 .. p0+B-1 for queries at
 *            tokens p0 .. p0+B-1)
 *   swa_len  [B] int32 device, each <= W: keys present in the window
 *   swa_tail 0: the present keys are the window's first swa_len rows (a
 *            ring that has not wrapped yet); 1: its last swa_len rows (a
 *            prefill window cut off at the start of the sequence)
 * Workspace: CSA2_OP_SPARSE_ATTN. */
CSA2_API int csa2_sparse_attn(const void* q, int32_t B, int32_t H, int32_t d,
                     const uint8_t* codes, const uint8_t* scales,
                     int64_t kv_seq_stride, int64_t n_cap, const int32_t* idx,
                     int32_t k, const void* swa, int64_t swa_seq_stride,
                     int32_t W, int32_t swa_tail, const int32_t* swa_len,
                     float softmax_scale,
                     void* out, void* ws, size_t ws_bytes, int32_t* d_status,
                     void* stream);

/* ---- a10+a11: one layer group [CSA2][TG] -------------------------------- */
enum csa2_mode { CSA2_MODE_FULL = 0, CSA2_MODE_REINDEX = 1 };
enum csa2_pool_rule { CSA2_POOL_NONE = 0, CSA2_POOL_MEAN_KEY = 1, CSA2_POOL_BLOCK_MAX = 2 };

/* Arguments of csa2_layer_group. Pointers are device pointers unless noted. */
typedef struct csa2_group_args {
  int32_t mode;          /* CSA2_MODE_FULL or CSA2_MODE_REINDEX               */
  int32_t n_reuse;       /* Reuse layers that follow the first layer          */
  int32_t form_pool;     /* also form the pool for later groups (csa2_pool_rule):
                            CSA2_POOL_MEAN_KEY scores the blocks' mean keys
                            with qI_pool (any mode); CSA2_POOL_BLOCK_MAX takes
                            the block maxima of this Full layer's scores     */
  int32_t B, H, d, H_I, d_I, k, W, P;
  int64_t n_max;         /* host bound on every n[b]                          */
  int64_t n_cap;         /* cache capacity (rows per sequence)                */
  const int64_t* n;      /* [B] visible positions                             */
  const uint8_t* codes;  /* [B][n_cap][d/2]                                   */
  const uint8_t* scales; /* [B][n_cap][d/16]                                  */
  const uint8_t* kI;     /* [B][n_cap][d_I]                                   */
  const uint8_t* kbar;   /* [B][ceil(n_cap/8)][d_I] (CSA2_POOL_MEAN_KEY only) */
  const uint8_t* qI;     /* [B][H_I][d_I] the first layer's indexer query     */
  const float* w;        /* [B][H_I]                                          */
  const uint8_t* qI_pool;/* pool-forming query (NULL = qI)                    */
  const float* w_pool;   /* (NULL = w)                                        */
  int32_t* pool;         /* [B][P]: written if form_pool, read if REINDEX     */
  int32_t* idx;          /* [B][k]: the group's Top-K (written)               */
  const void* const* q_layers;    /* HOST array [1+n_reuse] of [B][H][d] bf16 */
  const void* const* swa_layers;  /* HOST array [1+n_reuse] of [B][W][d] bf16 */
  const int32_t* swa_len;         /* [B]                                      */
  void* const* out_layers;        /* HOST array [1+n_reuse] of [B][H][d] bf16 */
  float softmax_scale;
  void* ws;              /* workspace, CSA2_OP_LAYER_GROUP                    */
  size_t ws_bytes;
  int32_t* d_status;     /* optional                                          */
  void* const* events;   /* optional HOST array of cudaEvent_t recorded on
                            the stream: [0] the indexer scan begins, [1] the
                            scan ends, [2] Top-K (and pool) done, [3 + l]
                            layer l's attention done. The scan is the Full
                            scan, the Reindex scan, or, in a Reindex group
                            that forms the pool, the block-mean scan (the
                            pool's Top-K and the Reindex scan then fall
                            between [1] and [2]). Up to 8 layers are
                            attended by one launch, so the events of the
                            layers in it are recorded together after it      */
  int32_t n_events;      /* length of `events` (0 = none)                     */
  int32_t rows_per_seq;  /* query rows per sequence, R (0 or 1: one). With
                            R > 1 (multi-token decode: R new tokens of each
                            sequence decoded in one step) B counts rows, and
                            row r reads the caches of sequence r / R (codes,
                            scales, kI, kbar have B / R sequences); n, qI, w,
                            pool, idx, swa_len, q and out stay per row; each
                            layer's SWA array holds W + R - 1 linear rows per
                            sequence (tokens p - W + 1 .. p + R - 1 for its
                            first new token p), row r's window is rows
                            r % R .. r % R + W - 1 of it, with its swa_len[r]
                            present keys at the window's end. B % R == 0,
                            R <= 64.                                          */
} csa2_group_args;

/* Run one CSA2 layer group: the first layer (Full: scan all positions,
 * Top-K, optionally form the pool; Reindex: rescore the pool, Top-K), then
 * attention for the first layer and each Reuse layer with the group's
 * Top-K, each with its own main Q and SWA KV. */
CSA2_API int csa2_layer_group(const csa2_group_args* args, void* stream);

/* ---- prefill chunk (encoder Full + Reuse layers) [CSA2][CED] ------------ */
/* Prefill indexer scores on the tensor cores: for every query q of a chunk
 * and every compressed entry j < n_keys (one cache shared by all queries),
 * scores[q][j] = sum_h w[q][h] * relu(qI[q][h] . kI[j]), FP8 E4M3 products
 * accumulated in fp32 (tcgen05 FP8 GEMM, TMA-fed). Entries past a query's
 * causal limit are scored too; the causal rule is applied by giving the
 * Top-K each query's visible count.
 *   qI [Q][8][128] u8; w [Q][8] fp32; kI [n_keys][128] u8
 *   scores [Q][scores_stride] fp32, scores_stride >= n_keys
 * Supported: H_I = 8, d_I = 128, n_keys <= 2^31 - 129, Q * 8 < 2^31. */
CSA2_API int csa2_prefill_index_scores(const uint8_t* qI, const float* w,
                                       int32_t Q, int32_t H_I, int32_t d_I,
                                       const uint8_t* kI, int64_t n_keys,
                                       float* scores, int64_t scores_stride,
                                       int32_t* d_status, void* stream);

/* Arguments of csa2_prefill_group. Pointers are device pointers unless noted. */
typedef struct csa2_prefill_args {
  int32_t Q;             /* queries (tokens) in the chunk                      */
  int32_t n_reuse;       /* Reuse layers after the Full layer                  */
  int32_t H, d, H_I, d_I, k, W;
  int64_t n_keys;        /* compressed main-KV entries in the shared cache     */
  const int64_t* n_vis;  /* [Q] entries visible to each query: an entry of
                            `ratio` tokens is visible once its last token is
                            at or before the query, i.e. floor((p+1)/ratio)   */
  const uint8_t* codes;  /* [n_keys][d/2]                                      */
  const uint8_t* scales; /* [n_keys][d/16]                                     */
  const uint8_t* kI;     /* [n_keys][d_I]                                      */
  const uint8_t* qI;     /* [Q][H_I][d_I]                                      */
  const float* w;        /* [Q][H_I]                                           */
  int32_t* idx;          /* [Q][k] Top-K of each query (written)               */
  const void* const* q_layers;    /* HOST array [1+n_reuse] of [Q][H][d] bf16 */
  const void* const* swa_layers;  /* HOST array [1+n_reuse] of the chunk's SWA
                                     rows [Q + W - 1][d] bf16: query q's window
                                     is rows q .. q + swa_len[q] - 1          */
  const int32_t* swa_len;         /* [Q] (<= W)                               */
  void* const* out_layers;        /* HOST array [1+n_reuse] of [Q][H][d] bf16 */
  float softmax_scale;
  void* ws;              /* workspace, CSA2_OP_PREFILL_GROUP                   */
  size_t ws_bytes;
  int32_t* d_status;     /* optional                                           */
  void* const* events;   /* optional HOST array of cudaEvent_t: [0] before the
                            indexer GEMM, [1] after it (its sampled pass,
                            the thresholds and the candidate-emitting pass),
                            [2] after Top-K, [3 + l] after layer l's
                            attention (recorded together for the up to 8
                            layers of one launch)                            */
  int32_t n_events;
} csa2_prefill_args;

/* One encoder group over a prefill chunk: Top-k of each query over its
 * visible entries by the indexer score of csa2_prefill_index_scores, then
 * sparse attention of the Full layer and of each Reuse layer with those
 * indices, every layer with its own Q and SWA rows.
 * The selection is fused into the tcgen05 indexer GEMM, and no score matrix
 * is written in the usual case: a GEMM pass over every 16th (or sparser)
 * entry tile gives each query a threshold (the r-th best sampled score, r
 * sized for about 2048 entries at or above it; every visible entry when a
 * query sees at most 8192), the full GEMM pass then emits only the entries
 * at or above it, and the exact Top-k is taken over those. A query with
 * fewer than min(k, visible) of them, or more than 8192, is selected from
 * its full score row instead, which the GEMM then writes for its tile of 32
 * queries. Entry tiles that no query of a tile can see are skipped. The
 * result is the same Top-k in every case (score descending, then position
 * ascending). Supported: n_keys <= 2^31 - 129. */
CSA2_API int csa2_prefill_group(const csa2_prefill_args* args, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H_ */
