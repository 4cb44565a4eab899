// C-ABI entry points of the InfiniteHiP sparse prefill: per-query-block selection
// (hip_prefill_select) and its conversion to the prefill kernel's lists
// (hip_prefill_lists).
#include <algorithm>
#include <cmath>

#include "api_common.h"
#include "launch.h"
#include "profile.h"

namespace dsa {
namespace {

constexpr int kBq = 64;

int check_pf_shape(const dsa_prefill_shape *s) {
  if (!s) return fail(DSA_ERR_INVALID_ARG, "shape is NULL");
  if (s->B < 1 || s->S < 1) return fail(DSA_ERR_INVALID_ARG, "B=%d / S=%d < 1", s->B, s->S);
  if (s->H_q < 1 || s->H_kv < 1 || s->H_q % s->H_kv != 0)
    return fail(DSA_ERR_INVALID_ARG, "H_q=%d must be a positive multiple of H_kv=%d", s->H_q, s->H_kv);
  if (s->D != 64 && s->D != 128) return fail(DSA_ERR_UNSUPPORTED, "D=%d not in {64, 128}", s->D);
  const int G = s->H_q / s->H_kv;
  if (s->H_kv > 8) return fail(DSA_ERR_UNSUPPORTED, "H_kv=%d > 8 (one cluster spans the KV heads)", s->H_kv);
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(DSA_ERR_UNSUPPORTED, "H_q/H_kv=%d not in {1, 2, 4, 8}", G);
  const long rows = static_cast<long>(s->B) * ((s->S + kBq - 1) / kBq);
  if (rows > 65535) return fail(DSA_ERR_UNSUPPORTED, "B * ceil(S/64) = %ld > 65535 query blocks", rows);
  return DSA_OK;
}

int check_pf_cfg(const dsa_prefill_shape *s, const dsa_hip_cfg *c) {
  if (!c) return fail(DSA_ERR_INVALID_ARG, "cfg is NULL");
  if (c->n_stages < 1 || c->n_stages > DSA_MAX_STAGES)
    return fail(DSA_ERR_INVALID_ARG, "n_stages=%d outside [1, %d]", c->n_stages, DSA_MAX_STAGES);
  if (c->n_sink < 0 || c->n_stream < 0) return fail(DSA_ERR_INVALID_ARG, "n_sink / n_stream negative");
  const int G = s->H_q / s->H_kv;
  for (int i = 0; i < c->n_stages; ++i) {
    if (c->chunk[i] < 1 || c->chunk[i] > 256)
      return fail(DSA_ERR_INVALID_ARG, "chunk[%d]=%d outside [1, 256]", i, c->chunk[i]);
    if (c->keep[i] < c->chunk[i] || (i > 0 && c->keep[i] > c->keep[i - 1]))
      return fail(DSA_ERR_INVALID_ARG, "keep[%d]=%d below chunk or above keep[%d]", i, c->keep[i], i - 1);
    if (c->keep[i] / c->chunk[i] > 16384)
      return fail(DSA_ERR_INVALID_ARG, "keep[%d]/chunk[%d] > 16384 chunks", i, i);
    if (prefill_score_smem(s->D, G, c->chunk[i], i > 0) > 200 * 1024)
      return fail(DSA_ERR_UNSUPPORTED, "stage %d needs too much shared memory", i);
  }
  if ((c->n_sink + kBq - 1) / kBq + (c->n_stream + kBq - 1) / kBq + 2 > 512)
    return fail(DSA_ERR_UNSUPPORTED, "n_sink + n_stream spans more than 512 key blocks");
  return DSA_OK;
}

int pf_max_chunks(const dsa_prefill_shape *s, const dsa_hip_cfg *c, int i) {
  if (i == 0) {
    const long n0 = std::max(0L, static_cast<long>(s->S) - c->n_stream - c->n_sink);
    return static_cast<int>((n0 + c->chunk[0] - 1) / c->chunk[0]);
  }
  return (c->keep[i - 1] + c->chunk[i] - 1) / c->chunk[i];
}

struct PfWs {
  int32_t *kv_rows;
  float *score[DSA_MAX_STAGES];
  int32_t *list[DSA_MAX_STAGES];
  int32_t *cnt[DSA_MAX_STAGES];
  size_t bytes;
};

PfWs pf_layout(const dsa_prefill_shape *s, const dsa_hip_cfg *c, void *base) {
  PfWs w{};
  Carve cv(base);
  const size_t R = static_cast<size_t>(s->B) * ((s->S + kBq - 1) / kBq);
  w.kv_rows = cv.take<int32_t>(R);
  for (int i = 0; i < c->n_stages; ++i) {
    w.score[i] = cv.take<float>(R * pf_max_chunks(s, c, i));
    if (i + 1 < c->n_stages) {
      w.list[i] = cv.take<int32_t>(R * c->keep[i]);
      w.cnt[i] = cv.take<int32_t>(R);
    }
  }
  w.bytes = cv.bytes();
  return w;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

int dsa_hip_prefill_max_chunks(const dsa_prefill_shape *shape, const dsa_hip_cfg *cfg, int stage,
                               int *n_chunks) {
  clear_error();
  int st = check_pf_shape(shape);
  if (st) return st;
  if ((st = check_pf_cfg(shape, cfg))) return st;
  if (stage < 0 || stage >= cfg->n_stages)
    return fail(DSA_ERR_INVALID_ARG, "stage=%d outside [0, %d)", stage, cfg->n_stages);
  if (!n_chunks) return fail(DSA_ERR_ALIGNMENT, "n_chunks is NULL");
  *n_chunks = pf_max_chunks(shape, cfg, stage);
  return DSA_OK;
}

int hip_prefill_select_workspace(const dsa_prefill_shape *shape, const dsa_hip_cfg *cfg,
                                 size_t *bytes) {
  clear_error();
  int st = check_pf_shape(shape);
  if (st) return st;
  if ((st = check_pf_cfg(shape, cfg))) return st;
  if (!bytes) return fail(DSA_ERR_ALIGNMENT, "bytes is NULL");
  *bytes = pf_layout(shape, cfg, nullptr).bytes;
  return DSA_OK;
}

int hip_prefill_select(const void *q, const void *k, const dsa_prefill_shape *shape,
                       const dsa_hip_cfg *cfg, int32_t *sel_idx, int32_t *sel_cnt,
                       const dsa_hip_debug *dbg, void *ws, size_t ws_bytes, void *stream) {
  clear_error();
  int st = check_pf_shape(shape);
  if (st) return st;
  if ((st = check_pf_cfg(shape, cfg))) return st;
  if (!aligned(q, 16) || !aligned(k, 16))
    return fail(DSA_ERR_ALIGNMENT, "q and k must be non-NULL and 16-byte aligned");
  if (!aligned(sel_idx, 16) || !aligned(sel_cnt, 4))
    return fail(DSA_ERR_ALIGNMENT, "sel_idx (16-byte) and sel_cnt (4-byte) must be aligned");
  const size_t need = pf_layout(shape, cfg, nullptr).bytes;
  if (ws_bytes < need || !aligned(ws, 16))
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes (16-byte aligned) needed, got %zu", need,
                ws_bytes);
  const PfWs w = pf_layout(shape, cfg, ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int n_qblk = (shape->S + kBq - 1) / kBq;
  const int R = shape->B * n_qblk;
  cudaError_t e = launch_prefill_rows(w.kv_rows, R, n_qblk, shape->S, s);
  if (e != cudaSuccess) return cuda_fail(e, "prefill rows launch");
  const int n = cfg->n_stages;
  for (int i = 0; i < n; ++i) {
    PfScoreArgs sa{};
    sa.q = q;
    sa.k = k;
    sa.B = shape->B;
    sa.S = shape->S;
    sa.H_q = shape->H_q;
    sa.H_kv = shape->H_kv;
    sa.D = shape->D;
    sa.n_qblk = n_qblk;
    sa.n_sink = cfg->n_sink;
    sa.n_stream = cfg->n_stream;
    sa.kv_rows = w.kv_rows;
    sa.in_idx = i == 0 ? nullptr : w.list[i - 1];
    sa.in_cnt = i == 0 ? nullptr : w.cnt[i - 1];
    sa.in_stride = i == 0 ? 0 : cfg->keep[i - 1];
    sa.L = cfg->chunk[i];
    sa.max_chunks = pf_max_chunks(shape, cfg, i);
    sa.stage = i;
    sa.score = (dbg && dbg->chunk_score[i]) ? dbg->chunk_score[i] : w.score[i];
    sa.dbg_rep = dbg ? dbg->rep[i] : nullptr;
    sa.dbg_rho = dbg ? dbg->rep_score[i] : nullptr;
    if ((e = launch_prefill_score(sa, s)) != cudaSuccess) return cuda_fail(e, "prefill stage score launch");

    StageTopkArgs ta{};
    ta.kv_len = w.kv_rows;
    ta.B = R;
    ta.T_max = shape->S;
    ta.n_sink = cfg->n_sink;
    ta.n_stream = cfg->n_stream;
    ta.in_idx = sa.in_idx;
    ta.in_cnt = sa.in_cnt;
    ta.in_stride = sa.in_stride;
    ta.L = cfg->chunk[i];
    ta.K = cfg->keep[i] / cfg->chunk[i];
    ta.max_chunks = sa.max_chunks;
    ta.score = sa.score;
    const bool last = i + 1 == n;
    ta.out_idx = last ? sel_idx : w.list[i];
    ta.out_cnt = last ? sel_cnt : w.cnt[i];
    ta.out_stride = cfg->keep[i];
    ta.dbg_idx = dbg ? dbg->stage_idx[i] : nullptr;
    ta.dbg_cnt = dbg ? dbg->stage_cnt[i] : nullptr;
    {
      ProfScope ps("prefill_stage_topk", s);
      e = launch_stage_topk(ta, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "prefill stage topk launch");
  }
  return DSA_OK;
}

int hip_prefill_lists(const dsa_prefill_shape *shape, const dsa_hip_cfg *cfg, const int32_t *sel_idx,
                      const int32_t *sel_cnt, int max_blk, int max_col, int32_t *blk_cnt,
                      int32_t *blk_idx, int32_t *col_cnt, int32_t *col_idx, void *stream) {
  clear_error();
  int st = check_pf_shape(shape);
  if (st) return st;
  if ((st = check_pf_cfg(shape, cfg))) return st;
  const int keep = cfg->keep[cfg->n_stages - 1];
  const int need_blk = (cfg->n_sink + kBq - 1) / kBq + (cfg->n_stream + kBq - 1) / kBq + 2;
  if (max_blk < need_blk)
    return fail(DSA_ERR_INVALID_ARG, "max_blk=%d < %d (sink and window blocks)", max_blk, need_blk);
  if (max_col < keep + 2 * (kBq - 1))
    return fail(DSA_ERR_INVALID_ARG, "max_col=%d < %d (selection + partial sink / window blocks)",
                max_col, keep + 2 * (kBq - 1));
  if (!aligned(sel_idx, 4) || !aligned(sel_cnt, 4) || !aligned(blk_cnt, 4) || !aligned(blk_idx, 4) ||
      !aligned(col_cnt, 4) || !aligned(col_idx, 4))
    return fail(DSA_ERR_ALIGNMENT, "arrays must be non-NULL and 4-byte aligned");
  PfListArgs a{};
  a.B = shape->B;
  a.S = shape->S;
  a.H_q = shape->H_q;
  a.n_qblk = (shape->S + kBq - 1) / kBq;
  a.n_sink = cfg->n_sink;
  a.n_stream = cfg->n_stream;
  a.sel_idx = sel_idx;
  a.sel_cnt = sel_cnt;
  a.keep = keep;
  a.max_blk = max_blk;
  a.max_col = max_col;
  a.blk_cnt = blk_cnt;
  a.blk_idx = blk_idx;
  a.col_cnt = col_cnt;
  a.col_idx = col_idx;
  cudaError_t e = launch_prefill_lists(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prefill lists launch");
  return DSA_OK;
}

}  // extern "C"
