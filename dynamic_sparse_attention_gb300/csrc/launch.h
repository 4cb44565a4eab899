// Internal launcher interface between the C-ABI layer (api.cpp) and the kernels.
// Arguments are validated by the caller; launchers only enqueue work.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dsa.h"

namespace dsa {

// The driver's tensor-map encoder (NULL if the driver offers none), and a 4-D TMA map
// (d, head, position, batch) of a [B, S, H, D] bf16 tensor with a box of 64 d x 1 head
// x `rows` positions, 128-byte swizzle (prefill_tc.cu).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
bool make_bshd_map(CUtensorMap *m, const void *base, int D, int H, int S, int B, int rows);

// Launch with programmatic stream serialization allowed: the grid may start while
// the stream's previous kernel drains (its CTAs then wait in grid_dep_wait()).
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// One pruning stage's chunk scoring (SelectRep tournament + max over heads).
struct StageScoreArgs {
  const void *q;          // [B, T_q, H_q, D]
  const void *k;          // [B, T_max, H_kv, D]
  const int32_t *kv_len;  // [B]
  int B, T_max, T_q, H_q, H_kv, D, dtype;
  int n_sink, n_stream;   // stage 0 (implicit candidate range) only
  const int32_t *in_idx;  // explicit input list [B, in_stride] (NULL for stage 0)
  const int32_t *in_cnt;  // [B]
  int in_stride;
  int L;                  // chunk size
  int max_chunks;         // row stride of score / rep arrays
  float *score;           // [B, max_chunks]
  int32_t *dbg_rep;       // [B, H_q, max_chunks] or NULL
  float *dbg_rho;         // [B, H_q, max_chunks] or NULL
};
cudaError_t launch_stage_score(const StageScoreArgs &a, cudaStream_t s);
// the same scores with the tournament probes on the tensor cores (stage_score_tc.cu):
// bf16 q and k, one query row, H_q / H_kv in {2, 4, 8}, H_kv <= 8, chunks of more
// than four tokens
bool stage_score_tc_ok(const StageScoreArgs &a);
cudaError_t launch_stage_score_tc(const StageScoreArgs &a, cudaStream_t s);

// Top-K chunks + assembly of the kept tokens.
struct StageTopkArgs {
  const int32_t *kv_len;
  int B, T_max;
  int n_sink, n_stream;
  const int32_t *in_idx;  // NULL for stage 0
  const int32_t *in_cnt;
  int in_stride;
  int L, K;               // chunk size, chunks kept
  int max_chunks;
  const float *score;     // [B, max_chunks]
  int32_t *out_idx;       // [B, out_stride]
  int32_t *out_cnt;       // [B]
  int out_stride;         // >= K * L
  int32_t *dbg_idx;       // optional copy of out_idx (stride out_stride)
  int32_t *dbg_cnt;
  // the selection's last kernel lets the next grid of the stream start at once (the
  // decode gathers its sink and window keys meanwhile and waits for the list)
  bool release_dependents;
};
cudaError_t launch_stage_topk(const StageTopkArgs &a, cudaStream_t s);

// Split-K decode over sink + selected + window keys, then the LSE merge.
struct DecodeArgs {
  const void *q, *k, *v;
  const int32_t *kv_len;
  const int32_t *sel_idx;
  const int32_t *sel_cnt;
  int max_sel, n_sink, n_stream;
  float scale;
  int B, T_max, T_q, H_q, H_kv, D, dtype;
  int n_split, keys_per_split;
  int fix_per, sel_per;   // cluster path: sink / window keys and selected slots per CTA
  bool cluster;           // plan path (see DecodePlan)
  float *part;            // [B, n_split, T_q, H_q, D + 2]
  void *out;
  float *lse;
};
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s);
// Host validation of a decode call and its arguments, everything but `part`
// (api_decode.cpp); *part_floats = the split-K partials the plan needs (0: none).
int decode_prepare(const void *q, const void *k, const void *v, const int32_t *kv_len,
                   const int32_t *sel_idx, const int32_t *sel_cnt, int max_sel, int n_sink,
                   int n_stream, float scale, const dsa_decode_shape *shape, void *out,
                   float *lse, DecodeArgs *args, size_t *part_floats);

// Decode plan shared by the workspace query and the launch.
//  * cluster path (cluster = true): one thread-block cluster of n_split CTAs per
//    (batch row, KV head), keys_per_split keys per CTA, tensor-core tiles, merged in
//    distributed shared memory; needs no workspace.  bf16 with R = (H_q/H_kv)*T_q
//    <= 16 query rows per KV head.
//  * split path: n_split CTAs per (b, g) write partials to the workspace, a second
//    kernel merges them.
struct DecodePlan {
  bool cluster;
  int n_split;
  int keys_per_split;
};
DecodePlan decode_plan(int B, int H_kv, int R, int D, int dtype, int a_max);
cudaError_t launch_decode_mma(const DecodeArgs &a, cudaStream_t s);
// workspace floats of the split path (0 on the cluster path)
size_t decode_ws_floats(const DecodePlan &p, int B, int T_q, int H_q, int D);

// The query heads an index builder writes (per-head pattern mixes); every head when
// `all`, else heads < 256 whose bit is set.
struct HeadSet {
  bool all = true;
  uint32_t bits[8] = {};
  __host__ __device__ bool has(int h) const {
    return all || (h < 256 && ((bits[h >> 5] >> (h & 31)) & 1u));
  }
};

// Vertical-slash index build.
struct VsArgs {
  const void *q, *k;
  int B, S, H_q, H_kv, D;
  int last_q, n_vertical, n_slash;
  float scale;
  int32_t *vertical, *slash, *blk_cnt, *blk_idx, *col_cnt, *col_idx;
  float *dbg_vsum, *dbg_ssum;
  // scratch
  float *row_m, *row_l;       // [B, H_q, 64] final row max / sum (base-2 logits)
  float *part_m, *part_l;     // [B, H_kv, n_split, G*64] per key-split row stats
  float *vsum, *ssum;         // [B, H_q, S] column sums / diagonal sums
  float *slash_part;          // [B, H_q, n_ktile, vs_tc_diag()] per key-tile diagonal sums
  int n_ktile;
  HeadSet heads;              // heads whose lists are written (the estimate covers all)
};
cudaError_t launch_vs_index(const VsArgs &a, cudaStream_t s);
// The estimate's two passes on tcgen05 (vs_tc.cu): row statistics, then column sums and
// per-128-key-tile diagonal partials (vs_tc_diag() offsets each), then their combine.
struct VsTcLaunch {
  const void *q, *k;
  int B, S, H_q, H_kv, D, last_q;
  float scale;
  float *part_m, *part_l;      // [B, H_kv, n_split0 * khalves, G * 64]
  float *row_m, *row_l;        // [B, H_q, 64]
  float *vsum, *ssum;          // [B, H_q, S]
  float *slash_part;           // [B, H_q, n_ktile1, vs_tc_diag()]
  HeadSet heads;               // heads whose slash sums are combined
};
int vs_tc_check(int D, int G);   // shape limits: DSA_OK or a status with the reason
int vs_tc_ready();               // the driver's tensor-map encoder is there (launch time)
int vs_tc_tile0(int G);          // keys per tile of the row-statistics pass
int vs_tc_khalves(int G);        // row-statistics partials per key run (key parts)
int vs_tc_tile1();               // keys per tile of the sums pass
int vs_tc_diag();                // diagonal partials per sums-pass tile (floats)
void vs_tc_plan(int B, int H_kv, int n_ktile, int *n_split, int *tiles_per_split);
cudaError_t launch_vs_tc(const VsTcLaunch &l, cudaStream_t s);
int vs_tc_device_error();        // the estimate's device error word (read and cleared)
// wait limits of the tensor-core kernels' bounded waits (0 on success)
int vs_tc_set_wait_limit(unsigned long long ns);
// check words of a checked build (DSA_CHECKS; read and cleared; 0 in normal builds)
int decode_check_word();
int decode_mma_check_word();
int hip_select_check_word();
int stage_tc_check_word();
int prefill_tc_check_word();
int prefill_tc_set_wait_limit(unsigned long long ns);

// Sparse prefill attention over tile / column lists.
struct PrefillArgs {
  const void *q, *k, *v;
  int B, S, H_q, H_kv, D;
  int max_blk, max_col;
  const int32_t *blk_cnt, *blk_idx, *col_cnt, *col_idx;
  float scale;
  void *out;
  float *lse;
};
// The tcgen05 kernel's own limits (D in {64, 128}, positive scale, the bitmaps of one
// query-block pair in shared memory, the driver's tensor-map encoder): DSA_OK, or a
// status with the reason in dsa_last_error().
int prefill_tc_check(const PrefillArgs &a);
cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t s);

// MInference A-shape block lists (static: the initial blocks plus a band ending at the
// diagonal block).
struct AshapeArgs {
  int BH, H_q, n_qblk, max_blk;
  HeadSet heads;
  int n_global_blk, n_local_blk;
  int32_t *blk_cnt, *blk_idx, *col_cnt;
};
cudaError_t launch_ashape(const AshapeArgs &a, cudaStream_t s);

// MInference Block-Sparse estimate: mean-pooled blocks, top-k_b key blocks per row.
struct BsArgs {
  const void *q, *k;
  int B, S, H_q, H_kv, D;
  int nb, k_b, max_blk;
  float scale;
  float *q_pool, *k_pool;   // scratch: q [B, H_q, nb, D], k transposed [B, H_kv, D, nb]
  float *dbg_q_pool, *dbg_k_pool, *dbg_scores;     // optional copies / [B, H_q, nb, nb]
  int32_t *blk_cnt, *blk_idx, *col_cnt;
  HeadSet heads;                                   // query heads pooled, scored and written
};
cudaError_t launch_block_sparse(const BsArgs &a, cudaStream_t s);
// query blocks per CTA of the scoring kernel (0: nb too large for shared memory)
int bs_rows_per_cta(int nb, int D);

// InfiniteHiP sparse prefill: one pruning stage's scores for query blocks of 64 rows
// (rows r = b * n_qblk + m); the cluster of a launch spans the H_kv KV heads.
struct PfScoreArgs {
  const void *q, *k;            // bf16 [B, S, H_q, D], [B, S, H_kv, D]
  int B, S, H_q, H_kv, D, n_qblk;
  int n_sink, n_stream;
  const int32_t *kv_rows;       // [R] keys each query block sees
  const int32_t *in_idx, *in_cnt;   // previous stage's lists per row (NULL: stage 0)
  int in_stride;
  int L, max_chunks;
  int stage;                    // index of the pruning stage (for timing names)
  float *score;                 // [R, max_chunks]
  int32_t *dbg_rep;             // optional [R, H_q, max_chunks]
  float *dbg_rho;
};
cudaError_t launch_prefill_score(const PfScoreArgs &a, cudaStream_t s);
cudaError_t launch_prefill_rows(int32_t *kv_rows, int R, int n_qblk, int S, cudaStream_t s);
size_t prefill_score_smem(int D, int G, int L, bool explicit_list);
// per-query-block selections -> prefill tile / column lists (shared by every head)
struct PfListArgs {
  int B, S, H_q, n_qblk, n_sink, n_stream;
  const int32_t *sel_idx, *sel_cnt;   // [R, keep], [R]
  int keep, max_blk, max_col;
  int32_t *blk_cnt, *blk_idx, *col_cnt, *col_idx;   // [B, H_q, n_qblk(, max)]
};
cudaError_t launch_prefill_lists(const PfListArgs &a, cudaStream_t s);

}  // namespace dsa
