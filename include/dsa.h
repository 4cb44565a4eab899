/*
 * dsa.h -- C ABI of the GB300 (sm_103a) dynamic sparse attention library (libdsa.so).
 *
 * Two halves of one hot path:
 *   decode : hip_select          -- InfiniteHiP hierarchical chunk pruning
 *            sparse_attn_decode  -- split-K online-softmax GQA decode over the
 *                                   sink + selected + window keys, with a merge
 *   prefill: vs_index_build      -- MInference vertical-slash estimate, top-k and
 *                                   conversion to per-query-block tile/column lists
 *            ashape_index_build  -- MInference A-shape lists (initial blocks + band)
 *            block_sparse_index_build -- MInference Block-Sparse estimate (mean-pooled
 *                                   blocks, top-k_b key blocks per query block)
 *            mixed_index_build   -- one of the three patterns per head
 *            hip_prefill_select  -- InfiniteHiP pruning per 64-row query block
 *            hip_prefill_lists   -- its sink / selection / window as prefill lists
 *            sparse_attn_prefill -- causal attention over those 64x64 tiles and
 *                                   gathered columns
 *
 * Conventions shared by every entry point
 *   - Tensor arguments are DEVICE pointers owned by the caller.  Layouts are
 *     row-major and contiguous ("bshd": batch, sequence, head, head-dim).
 *     q, k, v and out must be 16-byte aligned; int32/float arrays 4-byte aligned.
 *   - The library never allocates device memory and never synchronises.  Every
 *     call enqueues its kernels on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and returns at once.  Scratch memory, where needed, is the
 *     caller's `ws` buffer, whose size the matching *_workspace() call returns.
 *     Calls hold no state between them; two calls may run concurrently on
 *     different streams if their ws and output buffers differ.
 *   - No host synchronisation and fixed-size outputs: a decode step can be
 *     captured in a CUDA graph.
 *   - Return value: DSA_OK or a negative dsa_status.  On a validation failure
 *     nothing is launched and no output is touched; dsa_last_error() gives a
 *     message (thread-local).  DSA_ERR_CUDA reports a launch failure.
 *   - Device-side data (kv_len, counts, index lists) is not read by the host.
 *     Out-of-range values are clamped or skipped in the kernels (kv_len to
 *     [0, T_max], counts to [0, capacity], positions outside the row or the
 *     sequence skipped), never dereferenced.  A checked build (compiled with
 *     -DDSA_CHECKS=1, libdsa_checked.so) also records every such value it meets
 *     and dsa_device_error then returns DSA_ERR_DEVICE_CHECK.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_VERSION 1
#define DSA_MAX_STAGES 8

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = -1,  /* a shape, config or size is out of range */
  DSA_ERR_UNSUPPORTED = -2,  /* valid, but not built (dtype, head dim, block size) */
  DSA_ERR_WORKSPACE = -3,    /* ws missing or ws_bytes below the *_workspace() size */
  DSA_ERR_ALIGNMENT = -4,    /* a pointer is NULL or misaligned */
  DSA_ERR_CUDA = -5,         /* a kernel launch failed (message from the CUDA runtime) */
  DSA_ERR_DEVICE_CHECK = -6  /* checked builds: a kernel met out-of-range device data */
} dsa_status;

/* Element types of q / k / v (out has the type of q):
 *   DSA_BF16        bf16 q, k, v (raw bit patterns)
 *   DSA_F32         fp32 q, k, v
 *   DSA_BF16_FP8KV  bf16 q; k and v FP8 E4M3 codes, one byte per element (OCP E4M3:
 *                   bias 7, no infinity, S.1111.111 NaN); D = 128 and at most 16 query
 *                   rows per KV head ((H_q/H_kv) * T_q <= 16).  The InfiniteHiP
 *                   summary's throughput runs store the KV cache in this type.  A
 *                   per-tensor scale is the caller's: fold k's scale into `scale` and
 *                   multiply out by v's (lse then refers to the rescaled scores). */
typedef enum { DSA_BF16 = 0, DSA_F32 = 1, DSA_BF16_FP8KV = 2 } dsa_dtype;

/* ------------------------------------------------------------------ decode */

/* Shape of one batched decode step.
 *   q      [B, T_q, H_q, D]   the query block (T_q rows share one index set)
 *   k, v   [B, T_max, H_kv, D] the resident KV cache; row t of batch b is valid
 *                              for t < kv_len[b]
 * H_q % H_kv == 0; query head h reads KV head h / (H_q / H_kv).
 * D in {64, 128}; dtype one of dsa_dtype (DSA_BF16_FP8KV: D = 128 only). */
typedef struct {
  int B, T_max, T_q, H_q, H_kv, D;
  int dtype;
} dsa_decode_shape;

/* Pruning configuration: n_stages stages, stage i with chunk size l_c = chunk[i]
 * and token budget k = keep[i] (so it keeps K = keep[i] / chunk[i] chunks).
 * 1 <= chunk[i] <= 4096, chunk[i] <= keep[i], keep non-increasing,
 * keep[i] / chunk[i] <= 16384.  n_sink initial and n_stream newest tokens are
 * never pruned and are attended by sparse_attn_decode. */
typedef struct {
  int n_stages;
  int chunk[DSA_MAX_STAGES];
  int keep[DSA_MAX_STAGES];
  int n_sink, n_stream;
} dsa_hip_cfg;

/* Optional per-stage outputs for inspection; any pointer may be NULL.
 *   stage_idx[i]  [B, keep[i]]             token list after stage i, ascending, -1 padded
 *   stage_cnt[i]  [B]                      its length
 *   chunk_score[i][B, dsa_hip_max_chunks(i)] chunk scores s_j (fp32)
 *   rep[i]        [B, H_q, max_chunks(i)]  representative token of (head, chunk)
 *   rep_score[i]  [B, H_q, max_chunks(i)]  its score max_t q_t . k_rep (fp32)
 * Entries past a row's chunk count are left untouched. */
typedef struct {
  int32_t *stage_idx[DSA_MAX_STAGES];
  int32_t *stage_cnt[DSA_MAX_STAGES];
  float *chunk_score[DSA_MAX_STAGES];
  int32_t *rep[DSA_MAX_STAGES];
  float *rep_score[DSA_MAX_STAGES];
} dsa_hip_debug;

/* Upper bound on the chunk count of stage `stage` (host only). */
int dsa_hip_max_chunks(const dsa_decode_shape *shape, const dsa_hip_cfg *cfg, int stage,
                       int *n_chunks);

/* Bytes of scratch hip_select needs for this shape and config (host only). */
int hip_select_workspace(const dsa_decode_shape *shape, const dsa_hip_cfg *cfg, size_t *bytes);

/* hip_select -- hierarchical chunk pruning of the middle tokens.
 * Source: InfiniteHiP summary (arXiv 2502.08910), section 3.4, "Formal Mechanism
 * of a Single Pruning Stage" (Alg. 2), "The Representative Token Selection
 * Algorithm (SelectRep)" (Alg. 3), Alg. 1 line 1 (candidate range).
 * For every batch row b with T = kv_len[b]:
 *   I0 = [n_sink, T - n_stream); for each stage: split I into chunks of l_c,
 *   pick a representative per (query head, chunk) by the halving tournament
 *   (right half wins only on a strictly larger first-token score), score the
 *   chunk by the max over heads and query rows of q . k_rep (fp32 dot of the
 *   stored inputs), keep the K best chunks (ties -> smaller chunk index; all if
 *   there are at most K), and concatenate their tokens in ascending order.
 * Outputs: sel_idx [B, keep[n_stages-1]] final token list ascending, -1 padded;
 *          sel_cnt [B] its length.  dbg may be NULL.
 * The last kernel lets the next kernel of the stream start early (programmatic
 * dependent launch); a kernel that takes that start still waits for this one before
 * it reads sel_idx / sel_cnt (sparse_attn_decode does), and a kernel launched the
 * ordinary way starts after this call completes, as usual.
 * Errors: INVALID_ARG / UNSUPPORTED for shapes and configs, ALIGNMENT for
 * NULL/misaligned pointers, WORKSPACE if ws_bytes is short, CUDA on launch. */
int hip_select(const void *q, const void *k, const int32_t *kv_len,
               const dsa_decode_shape *shape, const dsa_hip_cfg *cfg,
               int32_t *sel_idx, int32_t *sel_cnt, const dsa_hip_debug *dbg,
               void *ws, size_t ws_bytes, void *stream);

/* hip_select_cached -- hip_select with per-stage mask caching (InfiniteHiP, section 3.4
 * "Sparse Attention Mask Caching"): pruning stage i is recomputed only when bit i of
 * `refresh` is set -- a decoding loop sets it when step % n_refresh[i] == 0 -- and a
 * stage that is not refreshed keeps the token list it produced on an earlier call.
 * A refreshed stage i > 0 starts from the list stage i-1 holds at that moment (just
 * recomputed, or cached); stage 0 always starts from the full candidate range of the
 * current kv_len.  Lists of stages 0..n_stages-2 live in `ws`, the last stage's in
 * sel_idx / sel_cnt, so all three must be the same buffers, unchanged by the caller,
 * from one call to the next; refresh = (1 << n_stages) - 1 is exactly hip_select and
 * refresh = 0 launches nothing.  Cached lists are not re-validated: positions read back
 * are clamped to [0, T_max) before any key row is read, and counts to [0, keep[i]], so
 * a workspace that holds no earlier selection gives a meaningless selection but never
 * an access outside k or ws.  A context that grew since stage 0 last ran keeps that
 * stage's candidates: tokens that left the streaming window in between are attended
 * again only after the next refresh of stage 0.
 * Errors as for hip_select; a bit at or above n_stages is INVALID_ARG. */
int hip_select_cached(const void *q, const void *k, const int32_t *kv_len,
                      const dsa_decode_shape *shape, const dsa_hip_cfg *cfg, uint32_t refresh,
                      int32_t *sel_idx, int32_t *sel_cnt, const dsa_hip_debug *dbg, void *ws,
                      size_t ws_bytes, void *stream);

/* Bytes of scratch sparse_attn_decode needs (split-K partials) (host only). */
int sparse_attn_decode_workspace(const dsa_decode_shape *shape, int max_sel, int n_sink,
                                 int n_stream, size_t *bytes);

/* sparse_attn_decode -- Flash-Decoding over the attended set of each row:
 *   A = [0, min(n_sink,T)) U sel_idx[b, 0:sel_cnt[b]] U [max(n_sink, T-n_stream), T)
 * out[b,t,h,:] = softmax_j(scale * q[b,t,h] . k[b,j,g]) v[b,j,g] over j in A,
 * lse[b,t,h] = natural-log sum of exp(scale * q . k) (NULL to skip).
 * Source: InfiniteHiP summary, section 3.4 "Block Sparse Attention
 * Implementation" (Flash Decoding with a final reduction) and "Formal
 * Background" (softmax attention); InfLLM guide, "Chunk-Level Attention Scoring
 * Engine" (softmax over sink U retrieved U local keys with 1/sqrt(d_k)).
 * sel_idx [B, max_sel] int32, entries ascending and inside [n_sink, T-n_stream);
 * sel_cnt [B] (clamped to [0, max_sel]).  out has the dtype of q.  A row with an
 * empty A gets out = 0 and lse = -inf.
 * Early start: the kernel is launched with programmatic stream serialization, so it
 * may start while the previous kernel of the stream still runs if that kernel allows
 * it (hip_select's last kernel does, at its start; ordinary kernels do not).  It then
 * reads q, k, v and kv_len and scores the sink and window keys at once, and waits for
 * the previous kernel before it reads sel_idx / sel_cnt or writes out / lse.  So a
 * kernel that writes q, k, v or kv_len and releases its dependents early must not come
 * right before this call on the stream.
 * Errors as for hip_select. */
int sparse_attn_decode(const void *q, const void *k, const void *v, const int32_t *kv_len,
                       const int32_t *sel_idx, const int32_t *sel_cnt, int max_sel, int n_sink,
                       int n_stream, float scale, const dsa_decode_shape *shape, void *out,
                       float *lse, void *ws, size_t ws_bytes, void *stream);

/* sparse_attn_decode_noalloc -- the same computation and arguments as
 * sparse_attn_decode, for callers that cannot allocate device memory when they
 * call it: a C runtime or plug-in with no device allocator of its own, or a
 * latency-bound loop that must not call cudaMalloc (which can synchronise the
 * device).  The pages have no counterpart; this is a packaging variant.
 * The split-K scratch is a fixed 4 MiB device array inside the library (held
 * on every GPU that loads the library until the process exits), so no `ws`
 * argument.  A call whose scratch (sparse_attn_decode_workspace) exceeds
 * 4 MiB is rejected with DSA_ERR_WORKSPACE and launches nothing.
 * The first call on a device looks up the array's device address (device
 * current at the call) and caches it for that device's current context; make
 * that first call before any stream capture.  After a cudaDeviceReset the
 * first call in the new context looks the address up again (the same rule:
 * not inside a capture).  All calls share the one array and nothing in it needs clearing
 * (each call overwrites the slots it reads), but calls that overlap on the
 * GPU (other streams, other threads) race on it: serialise them. */
int sparse_attn_decode_noalloc(const void *q, const void *k, const void *v,
                               const int32_t *kv_len, const int32_t *sel_idx,
                               const int32_t *sel_cnt, int max_sel, int n_sink, int n_stream,
                               float scale, const dsa_decode_shape *shape, void *out, float *lse,
                               void *stream);

/* ------------------------------------------------------------------ prefill */

/* Shape of one causal prefill: q/out [B, S, H_q, D], k/v [B, S, H_kv, D], bf16,
 * D in {64, 128}, H_q % H_kv == 0. */
typedef struct {
  int B, S, H_q, H_kv, D;
} dsa_prefill_shape;

/* Vertical-slash budgets: last_q estimate rows (<= 64 used: min(last_q, S)),
 * n_vertical columns and n_slash offsets kept per head (each <= S, >= 0),
 * tile size `block` (64 only). */
typedef struct {
  int last_q, n_vertical, n_slash, block;
} dsa_vs_cfg;

/* Optional estimate sums for inspection (NULL allowed): vsum / ssum [B, H_q, S]
 * fp32 column sums and slash (diagonal) sums of the estimated attention. */
typedef struct {
  float *vsum;
  float *ssum;
} dsa_vs_debug;

int vs_index_build_workspace(const dsa_prefill_shape *shape, const dsa_vs_cfg *cfg,
                             size_t *bytes);

/* vs_index_build -- MInference vertical-slash index for every (b, query head).
 * Source: MInference summary (arXiv 2407.02490), section 3.4 "Online Dynamic
 * Index Estimation: Vertical-Slash Heads" (Alg. 2 steps 1-4) and "Vertical-Slash
 * Hybrid Kernel" (Alg. 4, two-way merge).
 *   A~ = softmax(q[S-r:S] k^T / sqrt(D) + causal) for the r = min(last_q, S) last
 *   queries; vertical = top n_vertical column sums, slash = top n_slash diagonal
 *   sums (offset o = query pos - key pos), ties -> smaller index, both ascending.
 *   Conversion, per query block m (nominal rows 64m..64m+63): the key blocks that
 *   the slash segments [64m-o, 64m+63-o] touch (clipped at 0) form the block
 *   list; vertical columns <= 64m+63 outside those blocks form the column list.
 * Outputs (n_qblk = ceil(S/64)):
 *   vertical [B, H_q, n_vertical], slash [B, H_q, n_slash]   ascending
 *   blk_cnt [B, H_q, n_qblk], blk_idx [B, H_q, n_qblk, n_qblk] ascending key blocks
 *   col_cnt [B, H_q, n_qblk], col_idx [B, H_q, n_qblk, n_vertical] ascending keys
 * Unused tails of blk_idx / col_idx rows are left untouched.  dbg may be NULL. */
int vs_index_build(const void *q, const void *k, const dsa_prefill_shape *shape,
                   const dsa_vs_cfg *cfg, int32_t *vertical, int32_t *slash, int32_t *blk_cnt,
                   int32_t *blk_idx, int32_t *col_cnt, int32_t *col_idx,
                   const dsa_vs_debug *dbg, void *ws, size_t ws_bytes, void *stream);

/* ashape_index_build -- MInference A-shape lists for every (b, query head): query
 * block m attends the key blocks j <= m with j < n_global/64 (the initial tokens) or
 * m - j < n_local/64 (a band of blocks ending at the diagonal block), rows causal
 * inside the diagonal block.  Source: MInference summary, "The Three Sparse Patterns"
 * (A-Shape Pattern) and "Sparse GPU Kernel Implementations (Appendix C.4)" (A-Shape
 * Kernel).  The lists depend on the shape only (q and k are not read).
 *   n_global, n_local  token counts, non-negative multiples of `block` (64 only)
 *   blk_cnt [B, H_q, n_qblk], blk_idx [B, H_q, n_qblk, max_blk] ascending key blocks,
 *   col_cnt [B, H_q, n_qblk] all 0 (call sparse_attn_prefill with max_col = 0)
 * max_blk below min(n_qblk, n_global/64 + n_local/64) is INVALID_ARG.  Unused tails of
 * blk_idx rows are left untouched. */
int ashape_index_build(const dsa_prefill_shape *shape, int block, int n_global, int n_local,
                       int max_blk, int32_t *blk_cnt, int32_t *blk_idx, int32_t *col_cnt,
                       void *stream);

/* Optional Block-Sparse intermediates for inspection (each may be NULL):
 *   q_pool [B, H_q, n_qblk, D], k_pool [B, H_kv, n_qblk, D] fp32 mean-pooled blocks;
 *   scores [B, H_q, n_qblk, n_qblk] fp32 scaled block logits q~ . k~ / sqrt(D), written
 *   for key blocks j <= m only (small S: n_qblk^2 floats per head). */
typedef struct {
  float *q_pool;
  float *k_pool;
  float *scores;
} dsa_bs_debug;

int block_sparse_index_build_workspace(const dsa_prefill_shape *shape, int block,
                                       size_t *bytes);

/* block_sparse_index_build -- MInference Block-Sparse lists for every (b, query head).
 * Source: MInference summary, "Online Dynamic Index Estimation: Block-Sparse Heads
 * (Algorithm 3)", steps 1-4:
 *   q~ = MeanPooling(q, 64) per query head, k~ = MeanPooling(k, 64) per KV head (a
 *   ragged last block averages the tokens it has);
 *   A~ = softmax(q~ k~^T / sqrt(D) + block-causal mask), key blocks after the query
 *   block masked (the diagonal block stays);
 *   query block m keeps the min(k_b, m + 1) largest entries of its row (ties -> smaller
 *   block index), ascending.  Softmax is monotone along a row, so the kernels rank the
 *   fp32 logits; query head h uses KV head h / (H_q / H_kv).
 *   blk_cnt / blk_idx [B, H_q, n_qblk(, max_blk)], col_cnt all 0 (max_col = 0 in
 *   sparse_attn_prefill).
 * max_blk below min(k_b, n_qblk) is INVALID_ARG; S whose n_qblk block scores do not
 * fit one CTA's shared memory (S above about 2.08M at D = 128) is UNSUPPORTED.  dbg may be
 * NULL. */
int block_sparse_index_build(const void *q, const void *k, const dsa_prefill_shape *shape,
                             int block, int k_b, int max_blk, int32_t *blk_cnt, int32_t *blk_idx,
                             int32_t *col_cnt, const dsa_bs_debug *dbg, void *ws, size_t ws_bytes,
                             void *stream);

/* ------------------------------------------------- InfiniteHiP sparse prefill */

/* hip_prefill_select -- the pruning stages of hip_select for every query block of a
 * causal prefill: block m (rows 64m .. 64m+63 of batch row b, one "row" r = b * n_qblk + m
 * of the outputs, n_qblk = ceil(S/64)) prunes the keys before its end, T_m = min(S,
 * 64 (m+1)), with the chunk score the max over every query head and every row of the
 * block.  Source: InfiniteHiP summary, section 3.4 "Formal Mechanism of a Single
 * Pruning Stage" (Alg. 2, b_q = 64; steps 1-7), "The Representative Token Selection
 * Algorithm (SelectRep)", and "Prefill Latency Details" (chunked sparse prefill).
 * q [B, S, H_q, D], k [B, S, H_kv, D] bf16; cfg as for hip_select (chunk[i] <= 256).
 *   sel_idx [B * n_qblk, keep[n-1]] ascending key positions (-1 padded, 16-byte
 *   aligned), sel_cnt [B * n_qblk].
 * dbg (NULL allowed) as for hip_select with rows r in place of batch rows; its array
 * sizes come from dsa_hip_prefill_max_chunks.  H_kv <= 8, H_q / H_kv in {1, 2, 4, 8},
 * B * n_qblk <= 65535, D in {64, 128}; else UNSUPPORTED. */
int hip_prefill_select_workspace(const dsa_prefill_shape *shape, const dsa_hip_cfg *cfg,
                                 size_t *bytes);
int dsa_hip_prefill_max_chunks(const dsa_prefill_shape *shape, const dsa_hip_cfg *cfg, int stage,
                               int *n_chunks);
int hip_prefill_select(const void *q, const void *k, const dsa_prefill_shape *shape,
                       const dsa_hip_cfg *cfg, int32_t *sel_idx, int32_t *sel_cnt,
                       const dsa_hip_debug *dbg, void *ws, size_t ws_bytes, void *stream);

/* hip_prefill_lists -- each query block's attended set [0, min(n_sink, T_m)) U its
 * selection U [max(n_sink, T_m - n_stream), T_m) as sparse_attn_prefill lists (rows
 * attend only keys <= themselves there): the 64-key blocks wholly inside the sink or
 * the window are tiles, every other attended key a column (ascending); every head gets
 * the same lists.  Source: InfiniteHiP summary, "Block Sparse Attention Implementation"
 * (prefill attention over the selected keys) and "Important: Sink and Streaming Tokens
 * Are Never Pruned".
 *   blk_cnt / blk_idx [B, H_q, n_qblk(, max_blk)], col_cnt / col_idx likewise with
 *   max_col; max_blk >= ceil(n_sink/64) + ceil(n_stream/64) + 2 and
 *   max_col >= keep[n-1] + 126, else INVALID_ARG. */
int hip_prefill_lists(const dsa_prefill_shape *shape, const dsa_hip_cfg *cfg, const int32_t *sel_idx,
                      const int32_t *sel_cnt, int max_blk, int max_col, int32_t *blk_cnt,
                      int32_t *blk_idx, int32_t *col_cnt, int32_t *col_idx, void *stream);

/* Mixed per-head patterns: MInference assigns each attention head one of its three
 * patterns (MInference summary, "The Three Sparse Patterns"; the assignment itself
 * comes from an offline search that needs a model and is an input here). */
enum {
  DSA_PATTERN_VERTICAL_SLASH = 0,
  DSA_PATTERN_A_SHAPE = 1,
  DSA_PATTERN_BLOCK_SPARSE = 2
};

typedef struct {
  const uint8_t *head_pattern;  /* HOST array [H_q] of DSA_PATTERN_* (read during the call) */
  dsa_vs_cfg vs;                /* vertical-slash heads (block must be 64) */
  int n_global, n_local;        /* A-shape heads: token counts, multiples of 64 */
  int k_b;                      /* Block-Sparse heads */
} dsa_mixed_cfg;

int mixed_index_build_workspace(const dsa_prefill_shape *shape, const dsa_mixed_cfg *cfg,
                                size_t *bytes);

/* mixed_index_build -- every head's lists by its own pattern, into one set of arrays:
 * each head's rows are exactly what vs_index_build, ashape_index_build or
 * block_sparse_index_build writes for that head (the vertical-slash estimate still
 * runs over every head of a KV group that holds a vertical-slash head).
 *   blk_cnt [B, H_q, n_qblk], blk_idx [B, H_q, n_qblk, n_qblk] ascending key blocks,
 *   col_cnt [B, H_q, n_qblk] (0 for A-shape and Block-Sparse heads),
 *   col_idx [B, H_q, n_qblk, vs.n_vertical] (NULL allowed when no head is
 *   vertical-slash or vs.n_vertical = 0); pass max_blk = n_qblk and
 *   max_col = vs.n_vertical to sparse_attn_prefill.
 * H_q above 256 is UNSUPPORTED; a pattern value outside DSA_PATTERN_* and the checks
 * of each used pattern's own builder are INVALID_ARG / UNSUPPORTED as there. */
int mixed_index_build(const void *q, const void *k, const dsa_prefill_shape *shape,
                      const dsa_mixed_cfg *cfg, int32_t *blk_cnt, int32_t *blk_idx,
                      int32_t *col_cnt, int32_t *col_idx, void *ws, size_t ws_bytes,
                      void *stream);

/* sparse_attn_prefill -- causal attention of each query block over its listed
 * 64x64 key tiles, then its listed columns gathered 64 at a time, with one
 * online softmax.  Source: MInference summary, "Vertical-Slash Hybrid Kernel"
 * (Alg. 5) and "Block-Sparse FlashAttention Kernel (Appendix C.4.1)"; masked
 * attention of section 3.4 Eq. 1 with the mask constant as exact exclusion.
 * Row i of query block m attends key j <= i iff floor(j/64) is in
 * blk_idx[b,h,m,0:blk_cnt] or j is in col_idx[b,h,m,0:col_cnt].
 *   blk_idx [B, H_q, n_qblk, max_blk]  key-block ids, each < n_qblk, distinct
 *   col_idx [B, H_q, n_qblk, max_col]  key positions < S, distinct, not inside a
 *                                      listed block (else counted twice)
 * out [B, S, H_q, D] bf16; lse [B, H_q, S] fp32 natural log (NULL to skip).
 * A row with no attended key gets out = 0, lse = -inf.  block must be 64; scale
 * must be positive and finite (INVALID_ARG otherwise: the kernel orders scores by
 * their raw value).  S is bounded by the shared memory that holds the tile bitmaps
 * of one query-block pair (UNSUPPORTED beyond it). */
int sparse_attn_prefill(const void *q, const void *k, const void *v,
                        const dsa_prefill_shape *shape, int block, int max_blk, int max_col,
                        const int32_t *blk_cnt, const int32_t *blk_idx, const int32_t *col_cnt,
                        const int32_t *col_idx, float scale, void *out, float *lse,
                        void *stream);

/* ------------------------------------------------------------------ timing */

/* Per-kernel launch timing, off by default.  While enabled, every kernel the
 * library launches is bracketed by two CUDA events recorded on the call's own
 * stream (host-side bookkeeping only; nothing changes in the kernels).
 * dsa_profile_collect waits for the recorded events, returns one entry per
 * kernel name in first-launch order (name is a static string of the library),
 * writes min(n, max_out) entries and the total count to *n_out, and clears the
 * records.  Not a source-page operation: a measurement aid. */
typedef struct {
  const char *name;
  int launches;
  double total_ms;
} dsa_kernel_stat;

int dsa_profile_enable(int on);
int dsa_profile_collect(dsa_kernel_stat *out, int max_out, int *n_out);

/* ------------------------------------------------------------------ diagnostics */

/* Every wait inside the tensor-core kernels (the prefill attention and the two passes
 * of the vertical-slash estimate) is bounded; a CTA that gives up stops issuing work,
 * frees its resources and sets a device error word (the prefill CTA also writes zero
 * output).  dsa_device_error copies the words to *code (0 = none; bit 0: the prefill
 * attention, bit 1: the estimate; bit 2: in a checked build, a kernel met a kv_len,
 * count, selected position or list entry outside its documented range -- the call then
 * returns DSA_ERR_DEVICE_CHECK) and clears them.  It synchronises with the device
 * (cudaMemcpyFromSymbol); call it between steps, not on a hot path.  Not a
 * source-page operation. */
int dsa_device_error(int *code);

/* Sets the limit of those bounded waits to `ns` nanoseconds (0: back to the default of
 * half a second) for every later launch; it synchronises (cudaMemcpyToSymbol).  A test
 * aid: a limit of a few nanoseconds makes the waits run out, so that the give-up path
 * (stop, drain, free, error word) can be exercised without any fault.  Not a
 * source-page operation. */
int dsa_set_wait_limit(unsigned long long ns);

/* ------------------------------------------------------------------ helpers */

const char *dsa_last_error(void);   /* last validation / launch message of this thread */
const char *dsa_strerror(int status);
int dsa_version(void);              /* DSA_VERSION */

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
