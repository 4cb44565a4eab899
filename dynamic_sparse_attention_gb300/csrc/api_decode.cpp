// C-ABI entry points of the decode half: hip_select and sparse_attn_decode.
// Host-side validation, workspace layout and kernel launches on the caller's stream.
#include <cmath>

#include "api_common.h"
#include "launch.h"
#include "profile.h"

namespace dsa {
namespace {

const char *const kScoreNames[DSA_MAX_STAGES] = {
    "hip_stage_score_s0", "hip_stage_score_s1", "hip_stage_score_s2", "hip_stage_score_s3",
    "hip_stage_score_s4", "hip_stage_score_s5", "hip_stage_score_s6", "hip_stage_score_s7"};
const char *const kTopkNames[DSA_MAX_STAGES] = {
    "hip_stage_topk_s0", "hip_stage_topk_s1", "hip_stage_topk_s2", "hip_stage_topk_s3",
    "hip_stage_topk_s4", "hip_stage_topk_s5", "hip_stage_topk_s6", "hip_stage_topk_s7"};

int check_decode_shape(const dsa_decode_shape *s) {
  if (!s) return fail(DSA_ERR_INVALID_ARG, "shape is NULL");
  if (s->B < 1 || s->B > 65535) return fail(DSA_ERR_INVALID_ARG, "B=%d outside [1, 65535]", s->B);
  if (s->T_max < 1) return fail(DSA_ERR_INVALID_ARG, "T_max=%d < 1", s->T_max);
  if (s->T_q < 1) return fail(DSA_ERR_INVALID_ARG, "T_q=%d < 1", s->T_q);
  if (s->H_q < 1 || s->H_kv < 1 || s->H_q % s->H_kv != 0)
    return fail(DSA_ERR_INVALID_ARG, "H_q=%d must be a positive multiple of H_kv=%d", s->H_q, s->H_kv);
  if (s->H_q > 128) return fail(DSA_ERR_UNSUPPORTED, "H_q=%d > 128", s->H_q);
  if (s->D != 64 && s->D != 128) return fail(DSA_ERR_UNSUPPORTED, "D=%d not in {64, 128}", s->D);
  if (s->dtype != DSA_BF16 && s->dtype != DSA_F32 && s->dtype != DSA_BF16_FP8KV)
    return fail(DSA_ERR_UNSUPPORTED, "dtype=%d not DSA_BF16 / DSA_F32 / DSA_BF16_FP8KV", s->dtype);
  if (s->dtype == DSA_BF16_FP8KV && s->D != 128)
    return fail(DSA_ERR_UNSUPPORTED, "FP8 keys and values: D=%d, only 128", s->D);
  return DSA_OK;
}

int check_hip_cfg(const dsa_decode_shape *s, const dsa_hip_cfg *c) {
  if (!c) return fail(DSA_ERR_INVALID_ARG, "cfg is NULL");
  if (c->n_stages < 1 || c->n_stages > DSA_MAX_STAGES)
    return fail(DSA_ERR_INVALID_ARG, "n_stages=%d outside [1, %d]", c->n_stages, DSA_MAX_STAGES);
  if (c->n_sink < 0 || c->n_stream < 0)
    return fail(DSA_ERR_INVALID_ARG, "n_sink=%d / n_stream=%d negative", c->n_sink, c->n_stream);
  for (int i = 0; i < c->n_stages; ++i) {
    if (c->chunk[i] < 1 || c->chunk[i] > 4096)
      return fail(DSA_ERR_INVALID_ARG, "chunk[%d]=%d outside [1, 4096]", i, c->chunk[i]);
    if (c->keep[i] < c->chunk[i])
      return fail(DSA_ERR_INVALID_ARG, "keep[%d]=%d < chunk[%d]=%d", i, c->keep[i], i, c->chunk[i]);
    if (i > 0 && c->keep[i] > c->keep[i - 1])
      return fail(DSA_ERR_INVALID_ARG, "keep[%d]=%d > keep[%d]=%d (must not increase)", i,
                  c->keep[i], i - 1, c->keep[i - 1]);
    if (c->keep[i] / c->chunk[i] > 16384)
      return fail(DSA_ERR_INVALID_ARG, "keep[%d]/chunk[%d] = %d chunks > 16384", i, i,
                  c->keep[i] / c->chunk[i]);
  }
  if (s->T_q > 1) {
    const size_t qbytes = static_cast<size_t>(s->T_q) * s->H_q * s->D * 4;
    if (qbytes > 160 * 1024)
      return fail(DSA_ERR_UNSUPPORTED, "T_q*H_q*D*4 = %zu bytes of query block > 160 KiB", qbytes);
  }
  return DSA_OK;
}

int max_chunks(const dsa_decode_shape *s, const dsa_hip_cfg *c, int i) {
  long n_in;
  if (i == 0) {
    n_in = static_cast<long>(s->T_max) - c->n_sink - c->n_stream;
    if (n_in < 0) n_in = 0;
  } else {
    n_in = c->keep[i - 1];
  }
  return static_cast<int>((n_in + c->chunk[i] - 1) / c->chunk[i]);
}

struct HipWs {
  float *score[DSA_MAX_STAGES];
  int32_t *list[DSA_MAX_STAGES];
  int32_t *cnt[DSA_MAX_STAGES];
  size_t bytes;
};

HipWs hip_layout(const dsa_decode_shape *s, const dsa_hip_cfg *c, void *base) {
  HipWs w{};
  Carve cv(base);
  for (int i = 0; i < c->n_stages; ++i) {
    w.score[i] = cv.take<float>(static_cast<size_t>(s->B) * max_chunks(s, c, i));
    if (i + 1 < c->n_stages) {
      w.list[i] = cv.take<int32_t>(static_cast<size_t>(s->B) * c->keep[i]);
      w.cnt[i] = cv.take<int32_t>(s->B);
    }
  }
  w.bytes = cv.bytes();
  return w;
}

long attended_max(const dsa_decode_shape *s, int max_sel, int n_sink, int n_stream) {
  long a = static_cast<long>(n_sink < s->T_max ? n_sink : s->T_max) + max_sel +
           (n_stream < s->T_max ? n_stream : s->T_max);
  return a;
}

}  // namespace

// Validation and argument fill-in shared by sparse_attn_decode and
// sparse_attn_decode_noalloc; everything but the partials pointer.  *part_floats is the
// split-K scratch the plan needs (0 on the cluster path).
int decode_prepare(const void *q, const void *k, const void *v, const int32_t *kv_len,
                   const int32_t *sel_idx, const int32_t *sel_cnt, int max_sel, int n_sink,
                   int n_stream, float scale, const dsa_decode_shape *shape, void *out,
                   float *lse, DecodeArgs *args, size_t *part_floats) {
  int st = check_decode_shape(shape);
  if (st) return st;
  if (max_sel < 0 || n_sink < 0 || n_stream < 0)
    return fail(DSA_ERR_INVALID_ARG, "max_sel, n_sink and n_stream must be >= 0");
  if (!std::isfinite(scale)) return fail(DSA_ERR_INVALID_ARG, "scale is not finite");
  const int R = (shape->H_q / shape->H_kv) * shape->T_q;
  if (R * shape->D > 4096)
    return fail(DSA_ERR_UNSUPPORTED, "(H_q/H_kv)*T_q*D = %d > 4096 rows*dims per KV head", R * shape->D);
  if (shape->dtype == DSA_BF16_FP8KV && R > 16)
    return fail(DSA_ERR_UNSUPPORTED, "FP8 keys and values: (H_q/H_kv)*T_q = %d > 16", R);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return fail(DSA_ERR_ALIGNMENT, "q, k, v and out must be non-NULL and 16-byte aligned");
  if (!aligned(kv_len, 4) || !aligned(sel_cnt, 4) || (max_sel > 0 && !aligned(sel_idx, 4)))
    return fail(DSA_ERR_ALIGNMENT, "kv_len, sel_idx and sel_cnt must be non-NULL and 4-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(DSA_ERR_ALIGNMENT, "lse must be 4-byte aligned");
  const long a_max = attended_max(shape, max_sel, n_sink, n_stream);
  if (a_max > 0x7fffffffL) return fail(DSA_ERR_INVALID_ARG, "attended set too large");
  const DecodePlan plan = decode_plan(shape->B, shape->H_kv, R, shape->D, shape->dtype, static_cast<int>(a_max));
  if (plan.n_split > 65535) return fail(DSA_ERR_INVALID_ARG, "too many splits (%d)", plan.n_split);
  DecodeArgs &a = *args;
  a = DecodeArgs{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.kv_len = kv_len;
  a.sel_idx = sel_idx;
  a.sel_cnt = sel_cnt;
  a.max_sel = max_sel;
  a.n_sink = n_sink;
  a.n_stream = n_stream;
  a.scale = scale;
  a.B = shape->B;
  a.T_max = shape->T_max;
  a.T_q = shape->T_q;
  a.H_q = shape->H_q;
  a.H_kv = shape->H_kv;
  a.D = shape->D;
  a.dtype = shape->dtype;
  a.n_split = plan.n_split;
  a.keys_per_split = plan.keys_per_split;
  a.cluster = plan.cluster;
  a.part = nullptr;
  a.out = out;
  a.lse = lse;
  *part_floats = decode_ws_floats(plan, shape->B, shape->T_q, shape->H_q, shape->D);
  return DSA_OK;
}

}  // namespace dsa

using namespace dsa;

extern "C" {

int dsa_hip_max_chunks(const dsa_decode_shape *shape, const dsa_hip_cfg *cfg, int stage,
                       int *n_chunks) {
  clear_error();
  int st = check_decode_shape(shape);
  if (st) return st;
  if ((st = check_hip_cfg(shape, cfg))) return st;
  if (stage < 0 || stage >= cfg->n_stages)
    return fail(DSA_ERR_INVALID_ARG, "stage=%d outside [0, %d)", stage, cfg->n_stages);
  if (!n_chunks) return fail(DSA_ERR_ALIGNMENT, "n_chunks is NULL");
  *n_chunks = max_chunks(shape, cfg, stage);
  return DSA_OK;
}

int hip_select_workspace(const dsa_decode_shape *shape, const dsa_hip_cfg *cfg, size_t *bytes) {
  clear_error();
  int st = check_decode_shape(shape);
  if (st) return st;
  if ((st = check_hip_cfg(shape, cfg))) return st;
  if (!bytes) return fail(DSA_ERR_ALIGNMENT, "bytes is NULL");
  *bytes = hip_layout(shape, cfg, nullptr).bytes;
  return DSA_OK;
}

int hip_select_cached(const void *q, const void *k, const int32_t *kv_len,
                      const dsa_decode_shape *shape, const dsa_hip_cfg *cfg, uint32_t refresh,
                      int32_t *sel_idx, int32_t *sel_cnt, const dsa_hip_debug *dbg, void *ws,
                      size_t ws_bytes, void *stream) {
  clear_error();
  int st = check_decode_shape(shape);
  if (st) return st;
  if ((st = check_hip_cfg(shape, cfg))) return st;
  if (refresh >> cfg->n_stages)
    return fail(DSA_ERR_INVALID_ARG, "refresh mask 0x%x has bits at or above n_stages=%d", refresh,
                cfg->n_stages);
  if (!aligned(q, 16) || !aligned(k, 16))
    return fail(DSA_ERR_ALIGNMENT, "q and k must be non-NULL and 16-byte aligned");
  if (!aligned(kv_len, 4) || !aligned(sel_idx, 4) || !aligned(sel_cnt, 4))
    return fail(DSA_ERR_ALIGNMENT, "kv_len, sel_idx and sel_cnt must be non-NULL and 4-byte aligned");
  const size_t need = hip_layout(shape, cfg, nullptr).bytes;
  if (ws_bytes < need || (need > 0 && !aligned(ws, 16)))
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes (16-byte aligned) needed, got %zu", need,
                ws_bytes);
  const HipWs w = hip_layout(shape, cfg, ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int n = cfg->n_stages;
  for (int i = 0; i < n; ++i) {
    if (!((refresh >> i) & 1u)) continue;   // cached: the stage's list in ws (or sel_idx) stays
    const int maxc = max_chunks(shape, cfg, i);
    StageScoreArgs sa{};
    sa.q = q;
    sa.k = k;
    sa.kv_len = kv_len;
    sa.B = shape->B;
    sa.T_max = shape->T_max;
    sa.T_q = shape->T_q;
    sa.H_q = shape->H_q;
    sa.H_kv = shape->H_kv;
    sa.D = shape->D;
    sa.dtype = shape->dtype;
    sa.n_sink = cfg->n_sink;
    sa.n_stream = cfg->n_stream;
    sa.in_idx = i == 0 ? nullptr : w.list[i - 1];
    sa.in_cnt = i == 0 ? nullptr : w.cnt[i - 1];
    sa.in_stride = i == 0 ? 0 : cfg->keep[i - 1];
    sa.L = cfg->chunk[i];
    sa.max_chunks = maxc;
    sa.score = (dbg && dbg->chunk_score[i]) ? dbg->chunk_score[i] : w.score[i];
    sa.dbg_rep = dbg ? dbg->rep[i] : nullptr;
    sa.dbg_rho = dbg ? dbg->rep_score[i] : nullptr;
    cudaError_t e;
    {
      ProfScope ps(kScoreNames[i], s);
      e = launch_stage_score(sa, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "stage_score launch");

    StageTopkArgs ta{};
    ta.kv_len = kv_len;
    ta.B = shape->B;
    ta.T_max = shape->T_max;
    ta.n_sink = cfg->n_sink;
    ta.n_stream = cfg->n_stream;
    ta.in_idx = sa.in_idx;
    ta.in_cnt = sa.in_cnt;
    ta.in_stride = sa.in_stride;
    ta.L = cfg->chunk[i];
    ta.K = cfg->keep[i] / cfg->chunk[i];
    ta.max_chunks = maxc;
    ta.score = sa.score;
    const bool last = i + 1 == n;
    ta.out_idx = last ? sel_idx : w.list[i];
    ta.out_cnt = last ? sel_cnt : w.cnt[i];
    ta.out_stride = cfg->keep[i];
    ta.dbg_idx = dbg ? dbg->stage_idx[i] : nullptr;
    ta.dbg_cnt = dbg ? dbg->stage_cnt[i] : nullptr;
    ta.release_dependents = last;
    {
      ProfScope ps(kTopkNames[i], s);
      e = launch_stage_topk(ta, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "stage_topk launch");
  }
  return DSA_OK;
}

int hip_select(const void *q, const void *k, const int32_t *kv_len, const dsa_decode_shape *shape,
               const dsa_hip_cfg *cfg, int32_t *sel_idx, int32_t *sel_cnt,
               const dsa_hip_debug *dbg, void *ws, size_t ws_bytes, void *stream) {
  const bool ok = cfg && cfg->n_stages >= 1 && cfg->n_stages <= DSA_MAX_STAGES;
  const uint32_t all = ok ? (1u << cfg->n_stages) - 1u : 0u;   // a bad cfg fails in the callee
  return hip_select_cached(q, k, kv_len, shape, cfg, all, sel_idx, sel_cnt, dbg, ws, ws_bytes,
                           stream);
}

int sparse_attn_decode_workspace(const dsa_decode_shape *shape, int max_sel, int n_sink,
                                 int n_stream, size_t *bytes) {
  clear_error();
  int st = check_decode_shape(shape);
  if (st) return st;
  if (max_sel < 0 || n_sink < 0 || n_stream < 0)
    return fail(DSA_ERR_INVALID_ARG, "max_sel, n_sink and n_stream must be >= 0");
  if (!bytes) return fail(DSA_ERR_ALIGNMENT, "bytes is NULL");
  const long a_max = attended_max(shape, max_sel, n_sink, n_stream);
  if (a_max > 0x7fffffffL) return fail(DSA_ERR_INVALID_ARG, "attended set too large");
  const int R = (shape->H_q / shape->H_kv) * shape->T_q;
  if (shape->dtype == DSA_BF16_FP8KV && R > 16)
    return fail(DSA_ERR_UNSUPPORTED, "FP8 keys and values: (H_q/H_kv)*T_q = %d > 16", R);
  const DecodePlan plan = decode_plan(shape->B, shape->H_kv, R, shape->D, shape->dtype, static_cast<int>(a_max));
  const size_t nf = decode_ws_floats(plan, shape->B, shape->T_q, shape->H_q, shape->D);
  Carve cv(nullptr);
  if (nf) cv.take<float>(nf);
  *bytes = cv.bytes();
  return DSA_OK;
}

int sparse_attn_decode(const void *q, const void *k, const void *v, const int32_t *kv_len,
                       const int32_t *sel_idx, const int32_t *sel_cnt, int max_sel, int n_sink,
                       int n_stream, float scale, const dsa_decode_shape *shape, void *out,
                       float *lse, void *ws, size_t ws_bytes, void *stream) {
  clear_error();
  DecodeArgs a{};
  size_t nf = 0;
  int st = decode_prepare(q, k, v, kv_len, sel_idx, sel_cnt, max_sel, n_sink, n_stream, scale,
                          shape, out, lse, &a, &nf);
  if (st) return st;
  Carve cv(ws);
  a.part = nf ? cv.take<float>(nf) : nullptr;
  if (ws_bytes < cv.bytes() || (nf && !aligned(ws, 16)))
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes (16-byte aligned) needed, got %zu",
                cv.bytes(), ws_bytes);
  cudaError_t e = launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return DSA_OK;
}

}  // extern "C"
