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
#include <cooperative_groups.h>
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "profile.h"

namespace dsa {
namespace {

// Top-k of one row of n column sums or diagonal sums, ties -> smaller index, indices
// ascending.  One cluster of kTkC CTAs per row; CTA r owns a contiguous chunk of the row,
// copies its keys (order-preserving uint32 of the floats) into shared memory once
// (when the chunk fits; else every pass reads the row from L2), and then:
//   radix select, 12 + 12 + 8 bits from the top: per pass every CTA counts its chunk's
//   digits among the keys that match the prefix so far (shared-memory atomics; a warp
//   aggregation by __match_any_sync measured slower), CTA r merges bins [r * bins / kTkC, ...) of all CTAs' histograms
//   through distributed shared memory, and every CTA scans the merged histogram from
//   the top for the digit that holds the k-th largest key -- the same result in every
//   CTA;
//   compaction: warp w owns a contiguous run of the chunk and walks it 32 keys at a time
//   (lane l reads key 32 step + l), counting with ballots the keys above the threshold
//   and those equal to it; block and cluster prefix counts give each warp its first
//   output slot and its first equal-key rank, and a second walk writes the kept indices
//   (keys above, and equal keys of rank < k_eq) in index order.
constexpr int kTkC = 8;          // CTAs per row (one cluster)
constexpr int kTkNT = 512;       // threads per CTA
constexpr int kTkBins = 4096;
constexpr int kTkSmemKeys = 40 * 1024;   // keys staged per CTA at most (160 KB)

__device__ __forceinline__ uint32_t tk_block_scan(uint32_t v, uint32_t *s_w, uint32_t *total) {
  constexpr int NW = kTkNT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) s_w[warp] = incl;
  __syncthreads();
  const uint32_t x = lane < NW ? s_w[lane] : 0u;
  *total = __reduce_add_sync(kFull, x);
  const uint32_t before = __reduce_add_sync(kFull, lane < warp ? x : 0u);
  __syncthreads();   // s_w may be reused by the caller
  return before + incl;
}

__global__ void __cluster_dims__(kTkC, 1, 1) __launch_bounds__(kTkNT) vs_topk_kernel(VsArgs a, int staged) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ uint32_t s_hist[kTkBins];
  __shared__ uint32_t s_merged[kTkBins / kTkC];
  __shared__ uint32_t s_w[kTkNT / 32];
  __shared__ uint32_t s_res[4];
  extern __shared__ uint32_t s_keys[];   // [chunk] when staged
  const int rank = static_cast<int>(cluster.block_rank());
  const int bh = blockIdx.y;                   // b * H_q + h
  if (!a.heads.has(bh % a.H_q)) return;        // a head of another pattern (whole cluster)
  const bool is_slash = blockIdx.z == 1;
  const int S = a.S;
  const float *x = (is_slash ? a.ssum : a.vsum) + static_cast<size_t>(bh) * S;
  const int K = is_slash ? a.n_slash : a.n_vertical;
  int32_t *out = (is_slash ? a.slash : a.vertical) + static_cast<size_t>(bh) * K;
  if (K <= 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = (S + kTkC - 1) / kTkC;
  const int c_beg = min(S, rank * chunk), c_end = min(S, c_beg + chunk), n_c = c_end - c_beg;
  if (staged)
    for (int i = tid; i < n_c; i += kTkNT) s_keys[i] = ordered_key(x[c_beg + i]);
  __syncthreads();
  auto key_at = [&](int i) -> uint32_t {   // i relative to the chunk, < n_c
    return staged ? s_keys[i] : ordered_key(x[c_beg + i]);
  };
  const bool all = K >= S;
  uint32_t prefix = 0u, mask = 0u, k_rem = static_cast<uint32_t>(K);
  if (!all) {
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int sh = pass == 0 ? 20 : pass == 1 ? 8 : 0;
      const int width = pass == 2 ? 8 : 12;
      const uint32_t dmask = (1u << width) - 1u;
      const int nb = 1 << width;
      for (int i = tid; i < kTkBins; i += kTkNT) s_hist[i] = 0u;
      __syncthreads();
      for (int i0 = 0; i0 < n_c; i0 += kTkNT) {   // uniform trip count per CTA
        const int i = i0 + tid;
        const uint32_t key = i < n_c ? key_at(i) : 0u;
        const bool ok = i < n_c && (key & mask) == prefix;
        if (ok) atomicAdd(&s_hist[(key >> sh) & dmask], 1u);
      }
      cluster.sync();
      // this CTA's share of the bins, summed over the cluster in rank order
      const int per = nb / kTkC;
      for (int j = tid; j < per; j += kTkNT) {
        uint32_t sum = 0u;
#pragma unroll
        for (int c = 0; c < kTkC; ++c) sum += *cluster.map_shared_rank(&s_hist[rank * per + j], c);
        s_merged[j] = sum;
      }
      cluster.sync();
      // the merged counts from the top digit down: thread t holds digits nb-1-d_per t ..
      const int d_per = nb >= kTkNT ? nb / kTkNT : 1;
      uint32_t c8[8], sum8 = 0u;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int d = nb - 1 - tid * d_per - q;
        c8[q] = (q < d_per && d >= 0) ? *cluster.map_shared_rank(&s_merged[d % per], d / per) : 0u;
        sum8 += c8[q];
      }
      uint32_t total;
      const uint32_t incl = tk_block_scan(sum8, s_w, &total);
      if (incl - sum8 < k_rem && k_rem <= incl) {
        uint32_t run = incl - sum8;
        bool found = false;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (!found && q < d_per && run + c8[q] >= k_rem) {
            s_res[0] = static_cast<uint32_t>(nb - 1 - tid * d_per - q);
            s_res[1] = run;
            found = true;
          }
          run += c8[q];
        }
      }
      __syncthreads();
      prefix |= s_res[0] << sh;
      mask |= dmask << sh;
      k_rem -= s_res[1];
      cluster.sync();   // every CTA is done reading this pass's histograms
    }
  }
  const uint32_t thr = prefix, k_eq = k_rem;
  // compaction: warp w walks [w * wrun, (w + 1) * wrun) of the chunk, 32 keys a step
  constexpr int NW = kTkNT / 32;
  const int wrun = ((n_c + NW - 1) / NW + 31) & ~31;
  const int w_beg = min(n_c, warp * wrun), w_end = min(n_c, w_beg + wrun);
  const unsigned below = (1u << lane) - 1u;
  uint32_t n_gt = 0u, n_eq = 0u;
  for (int i0 = w_beg; i0 < w_end; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t key = i < w_end ? key_at(i) : 0u;
    const bool in = i < w_end;
    n_gt += __popc(__ballot_sync(kFull, in && (all || key > thr)));
    n_eq += __popc(__ballot_sync(kFull, in && !all && key == thr));
  }
  // per-warp totals -> block prefixes (one value per thread: lane 0 of each warp)
  uint32_t tot_gt, tot_eq;
  const uint32_t v_gt = lane == 0 ? n_gt : 0u, v_eq = lane == 0 ? n_eq : 0u;
  const uint32_t gt_incl = tk_block_scan(v_gt, s_w, &tot_gt);
  const uint32_t eq_incl = tk_block_scan(v_eq, s_w, &tot_eq);
  const uint32_t gt_warp = __shfl_sync(kFull, gt_incl - v_gt, 0);
  const uint32_t eq_warp = __shfl_sync(kFull, eq_incl - v_eq, 0);
  if (tid == 0) {
    s_res[2] = tot_gt;
    s_res[3] = tot_eq;
  }
  cluster.sync();
  uint32_t gt_before = 0u, eq_before = 0u;
  for (int c = 0; c < rank; ++c) {
    gt_before += *cluster.map_shared_rank(&s_res[2], c);
    eq_before += *cluster.map_shared_rank(&s_res[3], c);
  }
  cluster.sync();   // shared memory stays until every reader is done
  uint32_t eq_rank = eq_before + eq_warp;   // equal keys before this warp's run
  uint32_t slot = gt_before + gt_warp + (eq_rank < k_eq ? eq_rank : k_eq);
  for (int i0 = w_beg; i0 < w_end; i0 += 32) {
    const int i = i0 + lane;
    const bool in = i < w_end;
    const uint32_t key = in ? key_at(i) : 0u;
    const bool gt = in && (all || key > thr);
    const bool eq = in && !all && key == thr;
    const unsigned eq_b = __ballot_sync(kFull, eq);
    const bool keep = gt || (eq && eq_rank + __popc(eq_b & below) < k_eq);
    const unsigned keep_b = __ballot_sync(kFull, keep);
    if (keep) {
      const uint32_t sl = slot + __popc(keep_b & below);
      if (sl < static_cast<uint32_t>(K)) out[sl] = c_beg + i;
    }
    slot += __popc(keep_b);
    eq_rank += __popc(eq_b);
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
  // The slash list is ascending, so a thread's contiguous run of it touches few bitmap
  // words: the bits are gathered per word in a register and written with one atomicOr
  // per word (many threads or'ing into the same word serialise).
  const int32_t *slash = a.slash + bh * a.n_slash;
  {
    const int per = (a.n_slash + kConvNT - 1) / kConvNT;
    const int x0 = min(a.n_slash, tid * per), x1 = min(a.n_slash, x0 + per);
    int cur_w = -1;
    uint32_t cur_b = 0u;
    auto set = [&](int qd) {
      const int w = qd >> 5;
      if (w != cur_w) {
        if (cur_w >= 0 && cur_b) atomicOr(&s_bits[cur_w], cur_b);
        cur_w = w;
        cur_b = 0u;
      }
      cur_b |= 1u << (qd & 31);
    };
    for (int x = x0; x < x1; ++x) {
      const int o = slash[x];
      if (o < 0 || o >= a.S) continue;
      const int qd = o >> 6, r = o & 63;
      set(qd);
      if (r && qd + 1 < n_qblk) set(qd + 1);
    }
    if (cur_w >= 0 && cur_b) atomicOr(&s_bits[cur_w], cur_b);
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
    if ((n_qblk & 3) == 0) {
      // 16-byte stores: four consecutive entries per lane (rows start 16-byte aligned)
      int x = 4 * lane;
      for (; x + 3 < c_m; x += 128) {
        const int *dp = s_d + c_m - 1 - x;
        *reinterpret_cast<int4 *>(bl + x) = make_int4(m - dp[0], m - dp[-1], m - dp[-2], m - dp[-3]);
      }
      for (; x < c_m; ++x) bl[x] = m - s_d[c_m - 1 - x];   // at most one lane has a tail
    } else {
      for (int x = lane; x < c_m; x += 32) bl[x] = m - s_d[c_m - 1 - x];
    }
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
    dim3 g3(kTkC, a.B * a.H_q, 2);
    // keys staged in shared memory once (reading them from L2 in every pass instead
    // allows four CTAs per SM, one wave, but measured slower)
    const int chunk = (a.S + kTkC - 1) / kTkC;
    const int staged = chunk <= kTkSmemKeys ? 1 : 0;
    const size_t smem = staged ? static_cast<size_t>(chunk) * 4 : 0;
    if (smem > 0) {
      e = cudaFuncSetAttribute(vs_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    ProfScope ps("vs_topk", s);
    vs_topk_kernel<<<g3, kTkNT, smem, s>>>(a, staged);
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
