// MInference vertical-slash index build on sm_103a.
//
// Source: "MInference 1.0: Accelerating Pre-filling for Long-Context LLMs via Dynamic
// Sparse Attention" (paper-graph-ui summary), section 3.4 "Online Dynamic Index
// Estimation: Vertical-Slash Heads" (Alg. 2 steps 1-4) and "Vertical-Slash Hybrid
// Kernel" (Alg. 4, the two-way merge into block and column lists).
//
// Kernels, in launch order:
//   the estimate (vs_tc.cu): row statistics of the last r <= 64 queries of every head,
//                then the column sums and the per-tile diagonal partials of the
//                normalised probabilities, then their combine (tcgen05, deterministic);
//   vs_topk      per (batch, head, {vertical, slash}): radix select of the k largest
//                (ties -> smaller index) and an ascending compaction;
//   vs_convert   per (batch, head, run of query blocks): the slash offsets become a
//                bitmap of block diagonals d = m - n; block m lists n = m - d for every
//                d <= m, and keeps the vertical columns whose block is not listed.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "profile.h"

namespace dsa {
namespace {

constexpr int kTopkNT = 1024;

__global__ void __launch_bounds__(kTopkNT) vs_topk_kernel(VsArgs a) {
  constexpr int NT = kTopkNT;
  __shared__ uint32_t s_hist[256];
  __shared__ uint32_t s_res[2];
  __shared__ int s_warp[NT / 32 + 1];
  const int bh = blockIdx.x;                   // b * H_q + h
  if (!a.heads.has(bh % a.H_q)) return;        // a head of another pattern
  const bool is_slash = blockIdx.y == 1;
  const int S = a.S;
  const float *x = (is_slash ? a.ssum : a.vsum) + static_cast<size_t>(bh) * S;
  const int K = is_slash ? a.n_slash : a.n_vertical;
  int32_t *out = (is_slash ? a.slash : a.vertical) + static_cast<size_t>(bh) * K;
  if (K <= 0) return;
  uint32_t thr = 0;
  int k_eq = 0;
  const bool all = K >= S;
  if (!all)
    block_radix_select<NT>([&](int i) { return ordered_key(x[i]); }, S, K, s_hist, s_res, thr, k_eq);
  int eq_base = 0, keep_base = 0;
  for (int t0 = 0; t0 < S; t0 += NT) {
    const int i = t0 + threadIdx.x;
    const bool valid = i < S;
    const uint32_t key = (valid && !all) ? ordered_key(x[i]) : 0u;
    const bool is_eq = valid && !all && key == thr;
    int tot_eq, tot_keep;
    const int eq_rank = eq_base + block_flag_rank<NT>(is_eq, s_warp, &tot_eq);
    const bool kept = valid && (all || key > thr || (is_eq && eq_rank < k_eq));
    const int r = keep_base + block_flag_rank<NT>(kept, s_warp, &tot_keep);
    if (kept && r < K) out[r] = i;
    eq_base += tot_eq;
    keep_base += tot_keep;
  }
}

constexpr int kConvNT = 256;
constexpr int kConvRun = 64;   // query blocks per CTA

__global__ void __launch_bounds__(kConvNT) vs_convert_kernel(VsArgs a, int n_qblk) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int n_words = (n_qblk + 31) / 32;
  uint32_t *s_bits = reinterpret_cast<uint32_t *>(smem);
  int *s_wpre = reinterpret_cast<int *>(s_bits + n_words);
  int *s_d = s_wpre + n_words;
  int *s_vert = s_d + n_qblk;
  const int h = blockIdx.y, b = blockIdx.z;
  if (!a.heads.has(h)) return;   // a head of another pattern
  const size_t bh = static_cast<size_t>(b) * a.H_q + h;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int w = tid; w < n_words; w += kConvNT) s_bits[w] = 0u;
  __syncthreads();
  const int32_t *slash = a.slash + bh * a.n_slash;
  for (int x = tid; x < a.n_slash; x += kConvNT) {
    const int o = slash[x];
    if (o < 0 || o >= a.S) continue;
    const int qd = o >> 6, r = o & 63;
    atomicOr(&s_bits[qd >> 5], 1u << (qd & 31));
    if (r && qd + 1 < n_qblk) atomicOr(&s_bits[(qd + 1) >> 5], 1u << ((qd + 1) & 31));
  }
  const int32_t *vert = a.vertical + bh * a.n_vertical;
  for (int x = tid; x < a.n_vertical; x += kConvNT) s_vert[x] = vert[x];
  __syncthreads();
  if (warp == 0) {
    // exclusive prefix of word popcounts; lane owns a contiguous run of words
    const int per = (n_words + 31) / 32;
    const int w0 = lane * per, w1 = min(n_words, w0 + per);
    int sum = 0;
    for (int w = w0; w < w1; ++w) sum += __popc(s_bits[w]);
    int incl = sum;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int w = w0; w < w1; ++w) {
      s_wpre[w] = run;
      run += __popc(s_bits[w]);
    }
  }
  __syncthreads();
  for (int w = tid; w < n_words; w += kConvNT) {
    uint32_t bits = s_bits[w];
    int r = s_wpre[w];
    while (bits) {
      const int bit = __ffs(bits) - 1;
      s_d[r++] = w * 32 + bit;
      bits &= bits - 1;
    }
  }
  __syncthreads();
  const int m_begin = blockIdx.x * kConvRun;
  const int m_end = min(n_qblk, m_begin + kConvRun);
  for (int m = m_begin + warp; m < m_end; m += kConvNT / 32) {
    const int wm = m >> 5, bm = m & 31;
    const uint32_t below = bm == 31 ? 0xffffffffu : ((2u << bm) - 1u);
    const int c_m = s_wpre[wm] + __popc(s_bits[wm] & below);   // diagonals d <= m
    int32_t *bl = a.blk_idx + (bh * n_qblk + m) * static_cast<size_t>(n_qblk);
    for (int x = lane; x < c_m; x += 32) bl[x] = m - s_d[c_m - 1 - x];
    if (lane == 0) a.blk_cnt[bh * n_qblk + m] = c_m;
    int32_t *cl = a.col_idx + (bh * n_qblk + m) * static_cast<size_t>(a.n_vertical);
    int n_col = 0;
    const int row_end = m * 64 + 63;
    for (int x0 = 0; x0 < a.n_vertical; x0 += 32) {
      const int x = x0 + lane;
      const int j = x < a.n_vertical ? s_vert[x] : 0x7fffffff;
      bool keep = false;
      if (j >= 0 && j <= row_end) {
        const int d = m - (j >> 6);
        keep = !((s_bits[d >> 5] >> (d & 31)) & 1u);
      }
      const unsigned bal = __ballot_sync(kFull, keep);
      if (keep) cl[n_col + __popc(bal & ((1u << lane) - 1u))] = j;
      n_col += __popc(bal);
      if (__shfl_sync(kFull, j, 31) > row_end) break;   // vertical is ascending
    }
    if (lane == 0) a.col_cnt[bh * n_qblk + m] = n_col;
  }
}

cudaError_t launch_vs(const VsArgs &a, cudaStream_t s) {
  VsTcLaunch l;
  l.q = a.q;
  l.k = a.k;
  l.B = a.B;
  l.S = a.S;
  l.H_q = a.H_q;
  l.H_kv = a.H_kv;
  l.D = a.D;
  l.last_q = a.last_q;
  l.scale = a.scale;
  l.part_m = a.part_m;
  l.part_l = a.part_l;
  l.row_m = a.row_m;
  l.row_l = a.row_l;
  l.vsum = a.vsum;
  l.ssum = a.ssum;
  l.slash_part = a.slash_part;
  l.heads = a.heads;
  cudaError_t e = launch_vs_tc(l, s);
  if (e != cudaSuccess) return e;
  {
    dim3 g3(a.B * a.H_q, 2);
    ProfScope ps("vs_topk", s);
    vs_topk_kernel<<<g3, kTopkNT, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    const int n_qblk = (a.S + 63) / 64;
    const int n_words = (n_qblk + 31) / 32;
    const size_t smem = (2ull * n_words + n_qblk + a.n_vertical) * 4;
    e = cudaFuncSetAttribute(vs_convert_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 g4((n_qblk + kConvRun - 1) / kConvRun, a.H_q, a.B);
    ProfScope ps("vs_convert", s);
    vs_convert_kernel<<<g4, kConvNT, smem, s>>>(a, n_qblk);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_vs_index(const VsArgs &a, cudaStream_t s) { return launch_vs(a, s); }

}  // namespace dsa
