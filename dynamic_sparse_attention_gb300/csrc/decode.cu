// Sparse GQA decode on sm_103a: Flash-Decoding over the attended set
//   A = sink tokens U pruned selection U streaming window,
// split across CTAs along the key axis, each split producing (m, l, acc) partials,
// then an LSE merge.
//
// Source: "InfiniteHiP: Extending Language Model Context Up to 3 Million Tokens on a
// Single GPU" (paper-graph-ui summary), section 3.4 "Block Sparse Attention
// Implementation" (decoding: split the keys across thread blocks, partial softmax,
// final reduction) and "Formal Background" (softmax attention).  The InfLLM guide's
// "Chunk-Level Attention Scoring Engine" gives the same union-of-tiers softmax with
// a 1/sqrt(d_k) scale.
//
// Layout: the CTA serves all G query heads of KV head g and all T_q query rows at
// once, so each selected K/V row is gathered from HBM exactly once: 64-key tiles are
// staged into shared memory with 16-byte cp.async gathers (a token's row for head g
// is contiguous, 2*D bytes).
// This file holds the split path, for fp32 inputs and for more than 16 query rows
// per KV head: grid = (split, g, b) writes partials, a second kernel merges them.
// bf16 (or bf16 queries over FP8 keys and values) with at most 16 rows per KV head
// takes the tensor-core cluster kernel of
// decode_mma.cu.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "profile.h"

namespace dsa {

DSA_CHECK_WORD(decode_check_word)

namespace {

constexpr int kNT = 128;     // threads per split CTA
constexpr int kTK = 64;      // keys per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem_src));
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;\n" ::: "memory");
}

template <typename T, int D>
struct DecodeSmem {
  static constexpr int kPad = 16 / sizeof(T);     // 16-byte pad per K row (bank spread)
  static constexpr int kRowK = D + kPad;
  static size_t bytes(int R) {
    size_t o = 0;
    o += static_cast<size_t>(kTK) * kRowK * sizeof(T);   // s_k
    o += static_cast<size_t>(kTK) * D * sizeof(T);       // s_v
    o += static_cast<size_t>(R) * D * sizeof(float);     // s_q
    o += static_cast<size_t>(R) * kTK * sizeof(float);   // s_p
    o += static_cast<size_t>(kTK) * sizeof(int);         // s_pos
    o += static_cast<size_t>(3) * R * sizeof(float);     // s_m, s_l, s_alpha
    return o;
  }
};

template <typename T>
__device__ __forceinline__ float elem_to_f32(T x);
template <>
__device__ __forceinline__ float elem_to_f32<uint16_t>(uint16_t x) { return bf16_to_f32(x); }
template <>
__device__ __forceinline__ float elem_to_f32<float>(float x) { return x; }

// NACC = accumulators per thread (power of two, R*D <= NACC*kNT).
template <typename T, int D, int NACC>
__global__ void __launch_bounds__(kNT) decode_splitk_kernel(DecodeArgs a) {
  using SM = DecodeSmem<T, D>;
  extern __shared__ __align__(16) unsigned char smem[];
  const int G = a.H_q / a.H_kv;
  const int R = G * a.T_q;
  T *s_k = reinterpret_cast<T *>(smem);
  T *s_v = s_k + kTK * SM::kRowK;
  float *s_q = reinterpret_cast<float *>(s_v + kTK * D);
  float *s_p = s_q + R * D;
  int *s_pos = reinterpret_cast<int *>(s_p + R * kTK);
  float *s_m = reinterpret_cast<float *>(s_pos + kTK);
  float *s_l = s_m + R;
  float *s_alpha = s_l + R;

  grid_dep_wait();
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kv_raw = a.kv_len[b], cnt_raw = a.sel_cnt[b];
  DSA_CHECK(kv_raw >= 0 && kv_raw <= a.T_max);
  DSA_CHECK(cnt_raw >= 0 && cnt_raw <= a.max_sel);
  const int Tb = min(max(kv_raw, 0), a.T_max);
  const int n_s = min(a.n_sink, Tb);
  const int cnt = min(max(cnt_raw, 0), a.max_sel);
  const int w0 = max(a.n_sink, Tb - a.n_stream);
  const int n_w = max(0, Tb - w0);
  const int a_len = n_s + cnt + n_w;
  const int k_begin = split * a.keys_per_split;
  const int k_end = min(a_len, k_begin + a.keys_per_split);
  const int32_t *sel = a.sel_idx + static_cast<size_t>(b) * a.max_sel;
  const T *q = static_cast<const T *>(a.q);
  const T *kbase = static_cast<const T *>(a.k) + static_cast<size_t>(b) * a.T_max * a.H_kv * D +
                   static_cast<size_t>(g) * D;
  const T *vbase = static_cast<const T *>(a.v) + static_cast<size_t>(b) * a.T_max * a.H_kv * D +
                   static_cast<size_t>(g) * D;
  const size_t row_stride = static_cast<size_t>(a.H_kv) * D;
  const float sl2 = a.scale * kLog2e;

  // query rows r -> (t = r / G, h = g*G + r % G)
  for (int e = tid; e < R * D; e += kNT) {
    const int r = e / D, d = e - r * D;
    const int t = r / G, h = g * G + (r - t * G);
    s_q[e] = elem_to_f32<T>(q[((static_cast<size_t>(b) * a.T_q + t) * a.H_q + h) * D + d]);
  }
  for (int r = tid; r < R; r += kNT) {
    s_m[r] = -INFINITY;
    s_l[r] = 0.f;
  }
  float acc[NACC];
#pragma unroll
  for (int i = 0; i < NACC; ++i) acc[i] = 0.f;
  const int d_own = tid % D;
  const int r_step = kNT / D;           // rows advance by this between accumulators
  const int r_first = tid / D;
  __syncthreads();

  constexpr int CH = D * static_cast<int>(sizeof(T)) / 16;   // 16-byte pieces per row
  constexpr int EP = 16 / static_cast<int>(sizeof(T));       // elements per piece
  for (int kt = k_begin; kt < k_end; kt += kTK) {
    if (tid < kTK) {
      const int x = kt + tid;
      int pos = -1;
      if (x < k_end) {
        if (x < n_s) pos = x;
        else if (x < n_s + cnt) {
          pos = sel[x - n_s];
          DSA_CHECK(pos >= a.n_sink && pos < max(a.n_sink, Tb - a.n_stream));
        }
        else pos = w0 + (x - n_s - cnt);
        if (pos < 0 || pos >= Tb) pos = -1;   // never read outside the row's context
      }
      s_pos[tid] = pos;
    }
    __syncthreads();
    for (int e = tid; e < kTK * CH; e += kNT) {
      const int key = e / CH, c = e - key * CH;
      const int pos = s_pos[key];
      T *dk = s_k + key * SM::kRowK + c * EP;
      T *dv = s_v + key * D + c * EP;
      if (pos >= 0) {
        cp_async16(dk, kbase + static_cast<size_t>(pos) * row_stride + c * EP);
        cp_async16(dv, vbase + static_cast<size_t>(pos) * row_stride + c * EP);
      } else {
        *reinterpret_cast<uint4 *>(dk) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(dv) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_wait_all();
    __syncthreads();
    // scores (base-2 logits) for every (row, key) pair of the tile
    for (int e = tid; e < R * kTK; e += kNT) {
      const int r = e / kTK, key = e - r * kTK;
      float s = -INFINITY;
      if (s_pos[key] >= 0) {
        const float *qq = s_q + r * D;
        const T *kk = s_k + key * SM::kRowK;
        float dot = 0.f;
#pragma unroll 4
        for (int c = 0; c < CH; ++c) {
          float kf[EP];
          unpack16(*reinterpret_cast<const uint4 *>(kk + c * EP), kf, T());
#pragma unroll
          for (int u = 0; u < EP; ++u) dot = fmaf(qq[c * EP + u], kf[u], dot);
        }
        s = dot * sl2;
      }
      s_p[e] = s;
    }
    __syncthreads();
    // online softmax update, one warp per row
    for (int r = warp; r < R; r += kNT / 32) {
      const float x0 = s_p[r * kTK + lane], x1 = s_p[r * kTK + lane + 32];
      const float m_old = s_m[r];
      const float m_new = fmaxf(m_old, warp_max(fmaxf(x0, x1)));
      float p0 = 0.f, p1 = 0.f, alpha = 1.f;
      if (m_new != -INFINITY) {
        p0 = exp2f(x0 - m_new);
        p1 = exp2f(x1 - m_new);
        alpha = exp2f(m_old - m_new);
      }
      const float ls = warp_sum(p0 + p1);
      s_p[r * kTK + lane] = p0;
      s_p[r * kTK + lane + 32] = p1;
      if (lane == 0) {
        s_l[r] = s_l[r] * alpha + ls;
        s_m[r] = m_new;
        s_alpha[r] = alpha;
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NACC; ++i) {
      const int r = r_first + i * r_step;
      if (r < R) {
        float o = acc[i] * s_alpha[r];
        const float *pp = s_p + r * kTK;
#pragma unroll 8
        for (int key = 0; key < kTK; ++key) o = fmaf(pp[key], elem_to_f32<T>(s_v[key * D + d_own]), o);
        acc[i] = o;
      }
    }
    __syncthreads();
  }
  // partials: [B, n_split, T_q, H_q, D + 2]
#pragma unroll
  for (int i = 0; i < NACC; ++i) {
    const int r = r_first + i * r_step;
    if (r < R) {
      const int t = r / G, h = g * G + (r - t * G);
      float *P = a.part + ((((static_cast<size_t>(b) * a.n_split + split) * a.T_q + t) * a.H_q + h) *
                           (D + 2));
      P[d_own] = acc[i];
      if (d_own == 0) {
        P[D] = s_m[r];
        P[D + 1] = s_l[r];
      }
    }
  }
}

template <typename T, int D>
__global__ void decode_merge_kernel(DecodeArgs a) {
  grid_dep_wait();
  const int row = blockIdx.x;                 // (b, t, h)
  const int per_b = a.T_q * a.H_q;
  const int b = row / per_b, th = row - b * per_b;
  const size_t split_stride = static_cast<size_t>(per_b) * (D + 2);
  const float *P0 = a.part + (static_cast<size_t>(b) * a.n_split * per_b + th) * (D + 2);
  float M = -INFINITY;
  for (int s = 0; s < a.n_split; ++s) M = fmaxf(M, P0[s * split_stride + D]);
  float Lsum = 0.f, o = 0.f;
  const int d = threadIdx.x;
  if (M != -INFINITY) {
    for (int s = 0; s < a.n_split; ++s) {
      const float *P = P0 + s * split_stride;
      const float m = P[D];
      if (m == -INFINITY) continue;
      const float w = exp2f(m - M);
      Lsum = fmaf(P[D + 1], w, Lsum);
      o = fmaf(P[d], w, o);
    }
  }
  const float res = Lsum > 0.f ? o / Lsum : 0.f;
  const size_t out_off = static_cast<size_t>(row) * D + d;
  if constexpr (sizeof(T) == 2) static_cast<uint16_t *>(a.out)[out_off] = f32_to_bf16(res);
  else static_cast<float *>(a.out)[out_off] = res;
  if (a.lse && d == 0) a.lse[row] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
}

template <typename T, int D, int NACC>
cudaError_t launch_decode_t(const DecodeArgs &a, cudaStream_t s) {
  const int R = (a.H_q / a.H_kv) * a.T_q;
  const size_t smem = DecodeSmem<T, D>::bytes(R);
  auto kern = decode_splitk_kernel<T, D, NACC>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(a.n_split, a.H_kv, a.B);
  {
    ProfScope ps("decode_splitk", s);
    launch_pdl(kern, grid, dim3(kNT), smem, s, a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    ProfScope ps("decode_merge", s);
    launch_pdl(decode_merge_kernel<T, D>, dim3(a.B * a.T_q * a.H_q), dim3(D), 0, s, a);
  }
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_decode_d(const DecodeArgs &a, cudaStream_t s) {
  const int R = (a.H_q / a.H_kv) * a.T_q;
  const int need = (R * D + kNT - 1) / kNT;

  if (need <= 1) return launch_decode_t<T, D, 1>(a, s);
  if (need <= 2) return launch_decode_t<T, D, 2>(a, s);
  if (need <= 4) return launch_decode_t<T, D, 4>(a, s);
  if (need <= 8) return launch_decode_t<T, D, 8>(a, s);
  if (need <= 16) return launch_decode_t<T, D, 16>(a, s);
  return launch_decode_t<T, D, 32>(a, s);
}

}  // namespace

DecodePlan decode_plan(int B, int H_kv, int R, int D, int dtype, int a_max) {
  DecodePlan p{};
  if ((dtype == DSA_BF16 || dtype == DSA_BF16_FP8KV) && R <= 16) {
    // tensor-core cluster path: up to 16 CTAs per (b, g), whole 16-key sub-tiles each
    constexpr int kSub = 16;
    const int subs = a_max > 0 ? (a_max + kSub - 1) / kSub : 1;
    p.cluster = true;
    p.n_split = subs < 16 ? subs : 16;
    p.keys_per_split = ((subs + p.n_split - 1) / p.n_split) * kSub;
    return p;
  }
  // split path: about two CTAs per SM of a 152-SM part
  p.cluster = false;
  const int target = (304 + B * H_kv - 1) / (B * H_kv);
  int kps = (a_max + target - 1) / (target > 0 ? target : 1);
  kps = ((kps + kTK - 1) / kTK) * kTK;
  if (kps < kTK) kps = kTK;
  p.keys_per_split = kps;
  p.n_split = a_max > 0 ? (a_max + kps - 1) / kps : 1;
  return p;
}

size_t decode_ws_floats(const DecodePlan &p, int B, int T_q, int H_q, int D) {
  return p.cluster ? 0 : static_cast<size_t>(B) * p.n_split * T_q * H_q * (D + 2);
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s) {
  if (a.cluster) return launch_decode_mma(a, s);
  if (a.dtype == 0) return a.D == 128 ? launch_decode_d<uint16_t, 128>(a, s) : launch_decode_d<uint16_t, 64>(a, s);
  return a.D == 128 ? launch_decode_d<float, 128>(a, s) : launch_decode_d<float, 64>(a, s);
}

}  // namespace dsa
