// InfiniteHiP pruning stage on sm_103a: SelectRep tournaments + chunk score, then
// top-K chunk selection and index assembly.
//
// Source: "InfiniteHiP: Extending Language Model Context Up to 3 Million Tokens on a
// Single GPU" (paper-graph-ui summary), section 3.4: "Formal Mechanism of a Single
// Pruning Stage" (Alg. 2 steps 3-7) and "The Representative Token Selection Algorithm
// (SelectRep)" (Alg. 3).
//
// Layout of the scoring kernel: one CTA per (chunk j, batch row b); inside it, one
// 8-lane "octet" per query head h.  Each lane owns D/8 consecutive elements of the
// head dimension, so a key row (256 B at D=128 bf16) is fetched by the octet as
// contiguous 16-byte loads and the dot product closes with three xor-shuffles (the
// same value lands in all eight lanes, so every lane takes the same branch).  The
// tournament's left representative is always the current range start, whose score
// is already known; each iteration therefore loads exactly one new key row.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace dsa {
namespace {

struct InputRange {
  int n_in;            // number of candidate tokens
  int start;           // implicit range start (stage 0)
  const int32_t *in;   // explicit list or nullptr
};

__device__ __forceinline__ InputRange stage_input(const int32_t *kv_len, int b, int T_max,
                                                  int n_sink, int n_stream,
                                                  const int32_t *in_idx, const int32_t *in_cnt,
                                                  int in_stride) {
  InputRange r;
  if (in_idx == nullptr) {
    const int Tb = min(max(kv_len[b], 0), T_max);
    r.start = n_sink;
    r.n_in = max(0, Tb - n_stream - n_sink);
    r.in = nullptr;
  } else {
    r.start = 0;
    r.n_in = min(max(in_cnt[b], 0), in_stride);
    r.in = in_idx + static_cast<size_t>(b) * in_stride;
  }
  return r;
}

// smem layout shared with the host-side size computation below
__host__ __device__ inline size_t score_smem_pos_off() { return 128 * sizeof(float); }
__host__ __device__ inline size_t score_smem_q_off(bool explicit_list, int L) {
  size_t o = score_smem_pos_off() + (explicit_list ? ((static_cast<size_t>(L) + 3) & ~size_t(3)) * 4 : 0);
  return o;
}

template <typename T, int D, bool QREG>
__global__ void __launch_bounds__(1024) stage_score_kernel(StageScoreArgs a) {
  constexpr int EPL = D / 8;
  extern __shared__ __align__(16) unsigned char smem[];
  float *s_rho = reinterpret_cast<float *>(smem);
  int *s_pos = reinterpret_cast<int *>(smem + score_smem_pos_off());
  float *s_q = reinterpret_cast<float *>(smem + score_smem_q_off(a.in_idx != nullptr, a.L));

  const int b = blockIdx.y, j = blockIdx.x;
  const InputRange ir = stage_input(a.kv_len, b, a.T_max, a.n_sink, a.n_stream, a.in_idx,
                                    a.in_cnt, a.in_stride);
  const int n_chunk = (ir.n_in + a.L - 1) / a.L;
  if (j >= n_chunk) return;
  const int base = j * a.L;
  const int len = min(a.L, ir.n_in - base);
  const T *q = static_cast<const T *>(a.q) + static_cast<size_t>(b) * a.T_q * a.H_q * D;
  if (ir.in) {
    for (int x = threadIdx.x; x < len; x += blockDim.x) s_pos[x] = ir.in[base + x];
  }
  if (!QREG) {
    const int n = a.T_q * a.H_q * D;
    for (int e = threadIdx.x; e < n; e += blockDim.x) {
      if constexpr (sizeof(T) == 2) s_q[e] = bf16_to_f32(reinterpret_cast<const uint16_t *>(q)[e]);
      else s_q[e] = reinterpret_cast<const float *>(q)[e];
    }
  }
  __syncthreads();

  const int h = threadIdx.x >> 3, sub = threadIdx.x & 7;
  const int G = a.H_q / a.H_kv;
  if (h < a.H_q) {
    const int g = h / G;
    const unsigned omask = 0xffu << (threadIdx.x & 24);
    float qv[QREG ? EPL : 1];
    if (QREG) load_row<T, EPL>(q + static_cast<size_t>(h) * D + sub * EPL, qv);
    const T *kb = static_cast<const T *>(a.k) + static_cast<size_t>(b) * a.T_max * a.H_kv * D +
                  static_cast<size_t>(g) * D + sub * EPL;
    const size_t row_stride = static_cast<size_t>(a.H_kv) * D;
    const int T_q = QREG ? 1 : a.T_q;
    auto pos_of = [&](int x) -> int { return ir.in ? s_pos[x] : ir.start + base + x; };
    auto score = [&](int x) -> float {
      float kf[EPL];
      load_row<T, EPL>(kb + static_cast<size_t>(pos_of(x)) * row_stride, kf);
      float best = -INFINITY;
      for (int t = 0; t < T_q; ++t) {
        const float *qq = QREG ? qv : s_q + (static_cast<size_t>(t) * a.H_q + h) * D + sub * EPL;
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) d = fmaf(qq[e], kf[e], d);
        d += __shfl_xor_sync(omask, d, 4);
        d += __shfl_xor_sync(omask, d, 2);
        d += __shfl_xor_sync(omask, d, 1);
        best = fmaxf(best, d);
      }
      return best;
    };
    // SelectRep: halve [lo, hi] at the rounded-up midpoint; the right half wins only
    // when its first token scores strictly higher than the left half's first token.
    int lo = 0, hi = len - 1;
    float s_lo = score(0);
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      const float s_mid = score(mid);
      if (s_mid > s_lo) {
        lo = mid;
        s_lo = s_mid;
      } else {
        hi = mid - 1;
      }
    }
    if (sub == 0) {
      s_rho[h] = s_lo;
      if (a.dbg_rep) {
        const size_t o = (static_cast<size_t>(b) * a.H_q + h) * a.max_chunks + j;
        a.dbg_rep[o] = pos_of(lo);
        if (a.dbg_rho) a.dbg_rho[o] = s_lo;
      }
    }
  }
  __syncthreads();
  // chunk score: max over all query heads (and rows, already inside s_rho)
  if (threadIdx.x < 32) {
    float m = -INFINITY;
    for (int i = threadIdx.x; i < a.H_q; i += 32) m = fmaxf(m, s_rho[i]);
    m = warp_max(m);
    if (threadIdx.x == 0) a.score[static_cast<size_t>(b) * a.max_chunks + j] = m;
  }
}

constexpr int kTopkThreads = 1024;

__global__ void __launch_bounds__(kTopkThreads) stage_topk_kernel(StageTopkArgs a) {
  constexpr int NT = kTopkThreads;
  extern __shared__ int s_chunk_of_rank[];   // [K]
  __shared__ uint32_t s_hist[256];
  __shared__ uint32_t s_res[2];
  __shared__ int s_warp[NT / 32 + 1];
  const int b = blockIdx.x, tid = threadIdx.x;
  const InputRange ir = stage_input(a.kv_len, b, a.T_max, a.n_sink, a.n_stream, a.in_idx,
                                    a.in_cnt, a.in_stride);
  const int L = a.L;
  const int n_chunk = (ir.n_in + L - 1) / L;
  const float *sc = a.score + static_cast<size_t>(b) * a.max_chunks;
  const bool keep_all = n_chunk <= a.K;
  uint32_t thr = 0;
  int k_eq = 0;
  if (!keep_all) {
    // Top-K by score, ties -> smaller chunk index: find the K-th largest key, keep
    // everything above it and the first k_eq equal keys in index order.
    block_radix_select<NT>([&](int i) { return ordered_key(sc[i]); }, n_chunk, a.K, s_hist,
                           s_res, thr, k_eq);
  }
  int eq_base = 0, keep_base = 0;
  for (int t0 = 0; t0 < n_chunk; t0 += NT) {
    const int i = t0 + tid;
    const bool valid = i < n_chunk;
    const uint32_t key = (valid && !keep_all) ? ordered_key(sc[i]) : 0u;
    const bool is_eq = valid && !keep_all && key == thr;
    int tot_eq, tot_keep;
    const int eq_rank = eq_base + block_flag_rank<NT>(is_eq, s_warp, &tot_eq);
    const bool kept = valid && (keep_all || key > thr || (is_eq && eq_rank < k_eq));
    const int r = keep_base + block_flag_rank<NT>(kept, s_warp, &tot_keep);
    if (kept && r < a.K) s_chunk_of_rank[r] = i;
    eq_base += tot_eq;
    keep_base += tot_keep;
  }
  __syncthreads();
  const int n_kept = min(keep_base, max(a.K, 0));
  int count = n_kept * L;
  // only the last chunk of the list can be short; kept, it has the highest rank
  if (n_kept > 0 && s_chunk_of_rank[n_kept - 1] == n_chunk - 1) count -= n_chunk * L - ir.n_in;
  int32_t *out = a.out_idx + static_cast<size_t>(b) * a.out_stride;
  int32_t *dbg = a.dbg_idx ? a.dbg_idx + static_cast<size_t>(b) * a.out_stride : nullptr;
  for (int e = tid; e < a.out_stride; e += NT) {
    int val = -1;
    if (e < count) {
      const int r = e / L, x = e - r * L;
      const int src = s_chunk_of_rank[r] * L + x;
      val = ir.in ? ir.in[src] : ir.start + src;
    }
    out[e] = val;
    if (dbg) dbg[e] = val;
  }
  if (tid == 0) {
    a.out_cnt[b] = count;
    if (a.dbg_cnt) a.dbg_cnt[b] = count;
  }
}

template <typename T, int D>
cudaError_t launch_score_t(const StageScoreArgs &a, cudaStream_t s) {
  const bool explicit_list = a.in_idx != nullptr;
  const bool qreg = a.T_q == 1;
  size_t smem = score_smem_q_off(explicit_list, a.L);
  if (!qreg) smem += static_cast<size_t>(a.T_q) * a.H_q * D * sizeof(float);
  const int threads = ((8 * a.H_q + 31) / 32) * 32;
  dim3 grid(a.max_chunks, a.B);
  if (a.max_chunks == 0) return cudaSuccess;
  if (qreg) {
    auto kern = stage_score_kernel<T, D, true>;
    if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    kern<<<grid, threads, smem, s>>>(a);
  } else {
    auto kern = stage_score_kernel<T, D, false>;
    if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    kern<<<grid, threads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_stage_score(const StageScoreArgs &a, cudaStream_t s) {
  if (a.dtype == 0) {
    return a.D == 128 ? launch_score_t<uint16_t, 128>(a, s) : launch_score_t<uint16_t, 64>(a, s);
  }
  return a.D == 128 ? launch_score_t<float, 128>(a, s) : launch_score_t<float, 64>(a, s);
}

cudaError_t launch_stage_topk(const StageTopkArgs &a, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(a.K) * sizeof(int);
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(stage_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  stage_topk_kernel<<<a.B, kTopkThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dsa
