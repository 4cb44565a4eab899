// C-ABI entry points of the prefill half: vs_index_build, ashape_index_build,
// block_sparse_index_build and sparse_attn_prefill.
#include <algorithm>
#include <cmath>

#include "api_common.h"
#include "launch.h"

namespace dsa {
namespace {

constexpr int kBlock = 64;

int check_prefill_shape(const dsa_prefill_shape *s) {
  if (!s) return fail(DSA_ERR_INVALID_ARG, "shape is NULL");
  if (s->B < 1 || s->B > 65535) return fail(DSA_ERR_INVALID_ARG, "B=%d outside [1, 65535]", s->B);
  if (s->S < 1) return fail(DSA_ERR_INVALID_ARG, "S=%d < 1", s->S);
  if (s->H_q < 1 || s->H_kv < 1 || s->H_q % s->H_kv != 0)
    return fail(DSA_ERR_INVALID_ARG, "H_q=%d must be a positive multiple of H_kv=%d", s->H_q, s->H_kv);
  if (s->H_q > 65535) return fail(DSA_ERR_INVALID_ARG, "H_q=%d > 65535", s->H_q);
  if (s->D != 64 && s->D != 128) return fail(DSA_ERR_UNSUPPORTED, "D=%d not in {64, 128}", s->D);
  return DSA_OK;
}

int check_vs_cfg(const dsa_prefill_shape *s, const dsa_vs_cfg *c) {
  if (!c) return fail(DSA_ERR_INVALID_ARG, "cfg is NULL");
  if (c->block != kBlock) return fail(DSA_ERR_UNSUPPORTED, "block=%d (only 64)", c->block);
  if (c->last_q < 1 || c->last_q > 64)
    return fail(DSA_ERR_UNSUPPORTED, "last_q=%d outside [1, 64]", c->last_q);
  if (c->n_vertical < 0 || c->n_vertical > s->S)
    return fail(DSA_ERR_INVALID_ARG, "n_vertical=%d outside [0, S=%d]", c->n_vertical, s->S);
  if (c->n_slash < 0 || c->n_slash > s->S)
    return fail(DSA_ERR_INVALID_ARG, "n_slash=%d outside [0, S=%d]", c->n_slash, s->S);
  if (s->H_q / s->H_kv > 8)
    return fail(DSA_ERR_UNSUPPORTED, "H_q/H_kv=%d > 8 query heads per KV head", s->H_q / s->H_kv);
  int st = vs_tc_check(s->D, s->H_q / s->H_kv);
  if (st) return st;
  const long n_qblk = (s->S + kBlock - 1) / kBlock;
  const long conv_smem = (2 * ((n_qblk + 31) / 32) + n_qblk + c->n_vertical) * 4;
  if (conv_smem > 200 * 1024)
    return fail(DSA_ERR_UNSUPPORTED, "S=%d with n_vertical=%d needs %ld bytes of shared memory",
                s->S, c->n_vertical, conv_smem);
  return DSA_OK;
}

struct VsWs {
  float *part_m, *part_l, *row_m, *row_l, *vsum, *ssum, *slash_part;
  size_t bytes;
  int n_ktile, n_split;
};

VsWs vs_layout(const dsa_prefill_shape *s, void *base) {
  VsWs w{};
  Carve cv(base);
  const int G = s->H_q / s->H_kv;
  // row statistics: one partial per run of the first pass; diagonal partials: one set
  // per tile of the second pass
  const int tile0 = vs_tc_tile0(G), tile1 = vs_tc_tile1();
  int tps;
  vs_tc_plan(s->B, s->H_kv, (s->S + tile0 - 1) / tile0, &w.n_split, &tps);
  w.n_ktile = (s->S + tile1 - 1) / tile1;
  const size_t rows = static_cast<size_t>(s->B) * s->H_kv * w.n_split * vs_tc_khalves(G) * G * 64;
  w.part_m = cv.take<float>(rows);
  w.part_l = cv.take<float>(rows);
  w.row_m = cv.take<float>(static_cast<size_t>(s->B) * s->H_q * 64);
  w.row_l = cv.take<float>(static_cast<size_t>(s->B) * s->H_q * 64);
  w.vsum = cv.take<float>(static_cast<size_t>(s->B) * s->H_q * s->S);
  w.ssum = cv.take<float>(static_cast<size_t>(s->B) * s->H_q * s->S);
  w.slash_part = cv.take<float>(static_cast<size_t>(s->B) * s->H_q * w.n_ktile * vs_tc_diag());
  w.bytes = cv.bytes();
  return w;
}

struct BsWs {
  float *q_pool, *k_pool;
  size_t bytes;
};

BsWs bs_layout(const dsa_prefill_shape *s, void *base) {
  BsWs w{};
  Carve cv(base);
  const size_t nb = (s->S + kBlock - 1) / kBlock;
  w.q_pool = cv.take<float>(static_cast<size_t>(s->B) * s->H_q * nb * s->D);
  w.k_pool = cv.take<float>(static_cast<size_t>(s->B) * s->H_kv * nb * s->D);
  w.bytes = cv.bytes();
  return w;
}

cudaError_t run_vs(const void *q, const void *k, const dsa_prefill_shape *shape,
                   const dsa_vs_cfg *cfg, int32_t *vertical, int32_t *slash, int32_t *blk_cnt,
                   int32_t *blk_idx, int32_t *col_cnt, int32_t *col_idx, const dsa_vs_debug *dbg,
                   const VsWs &w, const HeadSet &heads, cudaStream_t stream) {
  VsArgs a{};
  a.q = q;
  a.k = k;
  a.B = shape->B;
  a.S = shape->S;
  a.H_q = shape->H_q;
  a.H_kv = shape->H_kv;
  a.D = shape->D;
  a.last_q = cfg->last_q;
  a.n_vertical = cfg->n_vertical;
  a.n_slash = cfg->n_slash;
  a.scale = 1.0f / std::sqrt(static_cast<float>(shape->D));
  a.vertical = vertical;
  a.slash = slash;
  a.blk_cnt = blk_cnt;
  a.blk_idx = blk_idx;
  a.col_cnt = col_cnt;
  a.col_idx = col_idx;
  a.row_m = w.row_m;
  a.row_l = w.row_l;
  a.part_m = w.part_m;
  a.part_l = w.part_l;
  a.vsum = (dbg && dbg->vsum) ? dbg->vsum : w.vsum;
  a.ssum = (dbg && dbg->ssum) ? dbg->ssum : w.ssum;
  a.slash_part = w.slash_part;
  a.n_ktile = w.n_ktile;
  a.heads = heads;
  return launch_vs_index(a, stream);
}

int check_ashape(const dsa_prefill_shape *shape, int n_global, int n_local, int max_blk) {
  if (n_global < 0 || n_local < 0 || n_global % kBlock || n_local % kBlock)
    return fail(DSA_ERR_INVALID_ARG, "n_global=%d / n_local=%d must be non-negative multiples of 64",
                n_global, n_local);
  const long n_qblk = (shape->S + kBlock - 1) / kBlock;
  const long need = std::min(n_qblk, static_cast<long>(n_global / kBlock) + n_local / kBlock);
  if (max_blk < need)
    return fail(DSA_ERR_INVALID_ARG, "max_blk=%d < %ld blocks per query block", max_blk, need);
  return DSA_OK;
}

cudaError_t run_ashape(const dsa_prefill_shape *shape, int n_global, int n_local, int max_blk,
                       int32_t *blk_cnt, int32_t *blk_idx, int32_t *col_cnt, const HeadSet &heads,
                       cudaStream_t stream) {
  AshapeArgs a{};
  a.BH = shape->B * shape->H_q;
  a.H_q = shape->H_q;
  a.n_qblk = (shape->S + kBlock - 1) / kBlock;
  a.max_blk = max_blk;
  a.n_global_blk = n_global / kBlock;
  a.n_local_blk = n_local / kBlock;
  a.blk_cnt = blk_cnt;
  a.blk_idx = blk_idx;
  a.col_cnt = col_cnt;
  a.heads = heads;
  return launch_ashape(a, stream);
}

int check_block_sparse(const dsa_prefill_shape *shape, int k_b, int max_blk) {
  const int nb = (shape->S + kBlock - 1) / kBlock;
  if (k_b < 0) return fail(DSA_ERR_INVALID_ARG, "k_b=%d < 0", k_b);
  if (max_blk < std::min(k_b, nb))
    return fail(DSA_ERR_INVALID_ARG, "max_blk=%d < min(k_b=%d, n_qblk=%d)", max_blk, k_b, nb);
  if (bs_rows_per_cta(nb, shape->D) < 1)
    return fail(DSA_ERR_UNSUPPORTED, "S=%d: a row of %d block scores exceeds shared memory",
                shape->S, nb);
  return DSA_OK;
}

cudaError_t run_block_sparse(const void *q, const void *k, const dsa_prefill_shape *shape, int k_b,
                             int max_blk, int32_t *blk_cnt, int32_t *blk_idx, int32_t *col_cnt,
                             const dsa_bs_debug *dbg, const BsWs &w, const HeadSet &heads,
                             cudaStream_t stream) {
  BsArgs a{};
  a.q = q;
  a.k = k;
  a.B = shape->B;
  a.S = shape->S;
  a.H_q = shape->H_q;
  a.H_kv = shape->H_kv;
  a.D = shape->D;
  a.nb = (shape->S + kBlock - 1) / kBlock;
  a.k_b = k_b;
  a.max_blk = max_blk;
  a.scale = 1.f / std::sqrt(static_cast<float>(shape->D));
  a.q_pool = w.q_pool;
  a.k_pool = w.k_pool;
  a.dbg_q_pool = dbg ? dbg->q_pool : nullptr;
  a.dbg_k_pool = dbg ? dbg->k_pool : nullptr;
  a.dbg_scores = dbg ? dbg->scores : nullptr;
  a.blk_cnt = blk_cnt;
  a.blk_idx = blk_idx;
  a.col_cnt = col_cnt;
  a.heads = heads;
  return launch_block_sparse(a, stream);
}

// Mixed per-head patterns: the vertical-slash scratch, its vertical / slash lists and
// the Block-Sparse pools, each only if some head uses that pattern.
struct MixedWs {
  VsWs vs;
  BsWs bs;
  int32_t *vertical, *slash;
  size_t bytes;
};

bool uses(const dsa_prefill_shape *s, const dsa_mixed_cfg *c, int pattern) {
  for (int h = 0; h < s->H_q; ++h)
    if (c->head_pattern[h] == pattern) return true;
  return false;
}

HeadSet heads_of(const dsa_prefill_shape *s, const dsa_mixed_cfg *c, int pattern) {
  HeadSet hs;
  hs.all = false;
  for (int h = 0; h < s->H_q; ++h)
    if (c->head_pattern[h] == pattern) hs.bits[h >> 5] |= 1u << (h & 31);
  return hs;
}

MixedWs mixed_layout(const dsa_prefill_shape *s, const dsa_mixed_cfg *c, void *base) {
  MixedWs w{};
  char *p = static_cast<char *>(base);
  size_t off = 0;
  if (uses(s, c, DSA_PATTERN_VERTICAL_SLASH)) {
    w.vs = vs_layout(s, p ? p + off : nullptr);
    off += w.vs.bytes;
    Carve cv(p ? p + off : nullptr);
    w.vertical = cv.take<int32_t>(static_cast<size_t>(s->B) * s->H_q * std::max(c->vs.n_vertical, 1));
    w.slash = cv.take<int32_t>(static_cast<size_t>(s->B) * s->H_q * std::max(c->vs.n_slash, 1));
    off += cv.bytes();
  }
  if (uses(s, c, DSA_PATTERN_BLOCK_SPARSE)) {
    w.bs = bs_layout(s, p ? p + off : nullptr);
    off += w.bs.bytes;
  }
  w.bytes = off;
  return w;
}

int check_mixed(const dsa_prefill_shape *s, const dsa_mixed_cfg *c) {
  if (!c || !c->head_pattern) return fail(DSA_ERR_INVALID_ARG, "cfg or cfg->head_pattern is NULL");
  if (s->H_q > 256) return fail(DSA_ERR_UNSUPPORTED, "H_q=%d > 256 heads for a pattern mix", s->H_q);
  for (int h = 0; h < s->H_q; ++h)
    if (c->head_pattern[h] > DSA_PATTERN_BLOCK_SPARSE)
      return fail(DSA_ERR_INVALID_ARG, "head_pattern[%d]=%d is not a pattern", h, c->head_pattern[h]);
  const int n_qblk = (s->S + kBlock - 1) / kBlock;
  int st;
  if (uses(s, c, DSA_PATTERN_VERTICAL_SLASH) && (st = check_vs_cfg(s, &c->vs))) return st;
  if (uses(s, c, DSA_PATTERN_A_SHAPE) && (st = check_ashape(s, c->n_global, c->n_local, n_qblk)))
    return st;
  if (uses(s, c, DSA_PATTERN_BLOCK_SPARSE) && (st = check_block_sparse(s, c->k_b, n_qblk))) return st;
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

int vs_index_build_workspace(const dsa_prefill_shape *shape, const dsa_vs_cfg *cfg, size_t *bytes) {
  clear_error();
  int st = check_prefill_shape(shape);
  if (st) return st;
  if ((st = check_vs_cfg(shape, cfg))) return st;
  if (!bytes) return fail(DSA_ERR_ALIGNMENT, "bytes is NULL");
  *bytes = vs_layout(shape, nullptr).bytes;
  return DSA_OK;
}

int vs_index_build(const void *q, const void *k, const dsa_prefill_shape *shape,
                   const dsa_vs_cfg *cfg, int32_t *vertical, int32_t *slash, int32_t *blk_cnt,
                   int32_t *blk_idx, int32_t *col_cnt, int32_t *col_idx,
                   const dsa_vs_debug *dbg, void *ws, size_t ws_bytes, void *stream) {
  clear_error();
  int st = check_prefill_shape(shape);
  if (st) return st;
  if ((st = check_vs_cfg(shape, cfg))) return st;
  if (!aligned(q, 16) || !aligned(k, 16))
    return fail(DSA_ERR_ALIGNMENT, "q and k must be non-NULL and 16-byte aligned");
  if ((cfg->n_vertical > 0 && (!aligned(vertical, 4) || !aligned(col_idx, 4))) ||
      (cfg->n_slash > 0 && !aligned(slash, 4)) || !aligned(blk_cnt, 4) || !aligned(blk_idx, 4) ||
      !aligned(col_cnt, 4))
    return fail(DSA_ERR_ALIGNMENT, "index outputs must be non-NULL and 4-byte aligned");
  if (dbg && ((dbg->vsum && !aligned(dbg->vsum, 4)) || (dbg->ssum && !aligned(dbg->ssum, 4))))
    return fail(DSA_ERR_ALIGNMENT, "debug sums must be 4-byte aligned");
  const VsWs need = vs_layout(shape, nullptr);
  if (ws_bytes < need.bytes || !aligned(ws, 16))
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes (16-byte aligned) needed, got %zu",
                need.bytes, ws_bytes);
  if ((st = vs_tc_ready())) return st;
  const VsWs w = vs_layout(shape, ws);
  cudaError_t e = run_vs(q, k, shape, cfg, vertical, slash, blk_cnt, blk_idx, col_cnt, col_idx, dbg,
                         w, HeadSet{}, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "vs_index_build launch");
  return DSA_OK;
}

int sparse_attn_prefill(const void *q, const void *k, const void *v,
                        const dsa_prefill_shape *shape, int block, int max_blk, int max_col,
                        const int32_t *blk_cnt, const int32_t *blk_idx, const int32_t *col_cnt,
                        const int32_t *col_idx, float scale, void *out, float *lse,
                        void *stream) {
  clear_error();
  int st = check_prefill_shape(shape);
  if (st) return st;
  if (block != kBlock) return fail(DSA_ERR_UNSUPPORTED, "block=%d (only 64)", block);
  if (max_blk < 0 || max_col < 0) return fail(DSA_ERR_INVALID_ARG, "max_blk / max_col negative");
  // the kernel orders scores by their raw value, which needs a positive scale
  if (!std::isfinite(scale) || !(scale > 0.f))
    return fail(DSA_ERR_INVALID_ARG, "scale=%g must be positive and finite", scale);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return fail(DSA_ERR_ALIGNMENT, "q, k, v and out must be non-NULL and 16-byte aligned");
  if (!aligned(blk_cnt, 4) || !aligned(col_cnt, 4) || (max_blk > 0 && !aligned(blk_idx, 4)) ||
      (max_col > 0 && !aligned(col_idx, 4)))
    return fail(DSA_ERR_ALIGNMENT, "list arrays must be non-NULL and 4-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(DSA_ERR_ALIGNMENT, "lse must be 4-byte aligned");
  PrefillArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.B = shape->B;
  a.S = shape->S;
  a.H_q = shape->H_q;
  a.H_kv = shape->H_kv;
  a.D = shape->D;
  a.max_blk = max_blk;
  a.max_col = max_col;
  a.blk_cnt = blk_cnt;
  a.blk_idx = blk_idx;
  a.col_cnt = col_cnt;
  a.col_idx = col_idx;
  a.scale = scale;
  a.out = out;
  a.lse = lse;
  if ((st = prefill_tc_check(a))) return st;
  cudaError_t e = launch_prefill_tc(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sparse_attn_prefill launch");
  return DSA_OK;
}

int ashape_index_build(const dsa_prefill_shape *shape, int block, int n_global, int n_local,
                       int max_blk, int32_t *blk_cnt, int32_t *blk_idx, int32_t *col_cnt,
                       void *stream) {
  clear_error();
  int st = check_prefill_shape(shape);
  if (st) return st;
  if (block != kBlock) return fail(DSA_ERR_UNSUPPORTED, "block=%d (only 64)", block);
  if ((st = check_ashape(shape, n_global, n_local, max_blk))) return st;
  if (!aligned(blk_cnt, 4) || !aligned(col_cnt, 4) || (max_blk > 0 && !aligned(blk_idx, 4)))
    return fail(DSA_ERR_ALIGNMENT, "list arrays must be non-NULL and 4-byte aligned");
  cudaError_t e = run_ashape(shape, n_global, n_local, max_blk, blk_cnt, blk_idx, col_cnt, HeadSet{},
                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ashape_index_build launch");
  return DSA_OK;
}

int block_sparse_index_build_workspace(const dsa_prefill_shape *shape, int block, size_t *bytes) {
  clear_error();
  int st = check_prefill_shape(shape);
  if (st) return st;
  if (block != kBlock) return fail(DSA_ERR_UNSUPPORTED, "block=%d (only 64)", block);
  if (!bytes) return fail(DSA_ERR_ALIGNMENT, "bytes is NULL");
  *bytes = bs_layout(shape, nullptr).bytes;
  return DSA_OK;
}

int block_sparse_index_build(const void *q, const void *k, const dsa_prefill_shape *shape,
                             int block, int k_b, int max_blk, int32_t *blk_cnt, int32_t *blk_idx,
                             int32_t *col_cnt, const dsa_bs_debug *dbg, void *ws, size_t ws_bytes,
                             void *stream) {
  clear_error();
  int st = check_prefill_shape(shape);
  if (st) return st;
  if (block != kBlock) return fail(DSA_ERR_UNSUPPORTED, "block=%d (only 64)", block);
  if ((st = check_block_sparse(shape, k_b, max_blk))) return st;
  if (!aligned(q, 16) || !aligned(k, 16))
    return fail(DSA_ERR_ALIGNMENT, "q and k must be non-NULL and 16-byte aligned");
  if (!aligned(blk_cnt, 4) || !aligned(col_cnt, 4) || (max_blk > 0 && !aligned(blk_idx, 4)))
    return fail(DSA_ERR_ALIGNMENT, "list arrays must be non-NULL and 4-byte aligned");
  if (dbg && ((dbg->q_pool && !aligned(dbg->q_pool, 16)) || (dbg->k_pool && !aligned(dbg->k_pool, 16)) ||
              (dbg->scores && !aligned(dbg->scores, 4))))
    return fail(DSA_ERR_ALIGNMENT, "debug arrays must be 16-byte (pools) / 4-byte aligned");
  const size_t need = bs_layout(shape, nullptr).bytes;
  if (ws_bytes < need || !aligned(ws, 16))
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes (16-byte aligned) needed, got %zu", need,
                ws_bytes);
  const BsWs w = bs_layout(shape, ws);
  cudaError_t e = run_block_sparse(q, k, shape, k_b, max_blk, blk_cnt, blk_idx, col_cnt, dbg, w,
                                   HeadSet{}, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "block_sparse_index_build launch");
  return DSA_OK;
}

int mixed_index_build_workspace(const dsa_prefill_shape *shape, const dsa_mixed_cfg *cfg,
                                size_t *bytes) {
  clear_error();
  int st = check_prefill_shape(shape);
  if (st) return st;
  if ((st = check_mixed(shape, cfg))) return st;
  if (!bytes) return fail(DSA_ERR_ALIGNMENT, "bytes is NULL");
  *bytes = mixed_layout(shape, cfg, nullptr).bytes;
  return DSA_OK;
}

int mixed_index_build(const void *q, const void *k, const dsa_prefill_shape *shape,
                      const dsa_mixed_cfg *cfg, int32_t *blk_cnt, int32_t *blk_idx,
                      int32_t *col_cnt, int32_t *col_idx, void *ws, size_t ws_bytes,
                      void *stream) {
  clear_error();
  int st = check_prefill_shape(shape);
  if (st) return st;
  if ((st = check_mixed(shape, cfg))) return st;
  const bool any_vs = uses(shape, cfg, DSA_PATTERN_VERTICAL_SLASH);
  if (!aligned(q, 16) || !aligned(k, 16))
    return fail(DSA_ERR_ALIGNMENT, "q and k must be non-NULL and 16-byte aligned");
  if (!aligned(blk_cnt, 4) || !aligned(blk_idx, 4) || !aligned(col_cnt, 4) ||
      (any_vs && cfg->vs.n_vertical > 0 && !aligned(col_idx, 4)))
    return fail(DSA_ERR_ALIGNMENT, "list arrays must be non-NULL and 4-byte aligned");
  const size_t need = mixed_layout(shape, cfg, nullptr).bytes;
  if (ws_bytes < need || (need > 0 && !aligned(ws, 16)))
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes (16-byte aligned) needed, got %zu", need,
                ws_bytes);
  if (any_vs && (st = vs_tc_ready())) return st;
  const MixedWs w = mixed_layout(shape, cfg, ws);
  const int n_qblk = (shape->S + kBlock - 1) / kBlock;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (uses(shape, cfg, DSA_PATTERN_A_SHAPE))
    e = run_ashape(shape, cfg->n_global, cfg->n_local, n_qblk, blk_cnt, blk_idx, col_cnt,
                   heads_of(shape, cfg, DSA_PATTERN_A_SHAPE), s);
  if (e == cudaSuccess && uses(shape, cfg, DSA_PATTERN_BLOCK_SPARSE))
    e = run_block_sparse(q, k, shape, cfg->k_b, n_qblk, blk_cnt, blk_idx, col_cnt, nullptr, w.bs,
                         heads_of(shape, cfg, DSA_PATTERN_BLOCK_SPARSE), s);
  if (e == cudaSuccess && any_vs)
    e = run_vs(q, k, shape, &cfg->vs, w.vertical, w.slash, blk_cnt, blk_idx, col_cnt, col_idx,
               nullptr, w.vs, heads_of(shape, cfg, DSA_PATTERN_VERTICAL_SLASH), s);
  if (e != cudaSuccess) return cuda_fail(e, "mixed_index_build launch");
  return DSA_OK;
}

}  // extern "C"
