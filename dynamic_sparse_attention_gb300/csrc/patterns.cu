// MInference A-shape and Block-Sparse head patterns as per-query-block key-block lists,
// the format sparse_attn_prefill consumes (no column entries).
//
// Source: "MInference 1.0: Accelerating Pre-filling for Long-Context LLMs via Dynamic
// Sparse Attention" (paper-graph-ui summary of arXiv 2407.02490): "The Three Sparse
// Patterns" (A-Shape Pattern), "Sparse GPU Kernel Implementations (Appendix C.4)"
// (A-Shape Kernel: the initial blocks plus a band of blocks ending at the diagonal) and
// "Online Dynamic Index Estimation: Block-Sparse Heads (Algorithm 3)":
//   Q~ = MeanPooling(Q, 64), K~ = MeanPooling(K, 64),
//   A~ = softmax(Q~ K~^T / sqrt(d) + block-causal mask), i_b = top-k_b of each row.
//
// A-shape: one warp per (b, h, query block) writes its list; the lists do not depend
// on the input.
//
// Block-Sparse, two kernels:
//  * bs_pool_kernel: one CTA per (b, 64-token block); each thread owns one 16-byte
//    piece (8 head dimensions of one head) of the token rows, so every load of a token
//    row is coalesced across the CTA, and sums it over the block's tokens in fp32.  Q
//    and K are each read once: this kernel is the HBM-bound part.
//    The pooled keys are stored transposed ([D][nb] per KV head) for the next kernel.
//  * bs_topk_kernel: one CTA per (b, query head, R consecutive query blocks).  The R
//    pooled query rows (pre-scaled) sit in shared memory; each thread scores two key
//    blocks against all R rows with fp32 FMAs, reading the keys' transposed columns
//    straight from L2 (coalesced across the warp: 4 FMAs per shared-memory load), and
//    the rows' scores stay in shared memory.  Then one warp per row finds the k_b-th
//    largest score (value buckets between the row's min and max, exact ranking inside
//    the boundary bucket, an 8-bit radix select when that bucket is crowded) and
//    writes the kept blocks in ascending order (larger score first, ties -> smaller
//    block index).  Softmax is monotone along a row, so the kernel ranks the scaled
//    logits; the causal mask is the row length m + 1.
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "profile.h"

namespace dsa {
namespace {

constexpr int kBlk = 64;

// ------------------------------------------------------------------------------ A-shape

__global__ void __launch_bounds__(256) ashape_kernel(AshapeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x * 8 + warp;
  if (m >= a.n_qblk) return;
  if (!a.heads.has(static_cast<int>(blockIdx.y) % a.H_q)) return;
  const size_t row = static_cast<size_t>(blockIdx.y) * a.n_qblk + m;
  const int n_init = min(a.n_global_blk, m + 1);             // blocks 0 .. n_init - 1
  const int band_lo = max(n_init, m - a.n_local_blk + 1);     // band blocks band_lo .. m
  const int cnt = n_init + max(0, m - band_lo + 1);
  int32_t *out = a.blk_idx + row * a.max_blk;
  for (int e = lane; e < cnt; e += 32) out[e] = e < n_init ? e : band_lo + (e - n_init);
  if (lane == 0) {
    a.blk_cnt[row] = cnt;
    a.col_cnt[row] = 0;
  }
}

// ------------------------------------------------------------------------------ pooling

constexpr int kPoolThreads = 512;

__global__ void __launch_bounds__(kPoolThreads) bs_pool_kernel(BsArgs a) {
  const int j = blockIdx.x, b = blockIdx.y;
  const int t0 = j * kBlk;
  const int rows = min(kBlk, a.S - t0);
  const float inv = 1.f / static_cast<float>(rows);
  const int pq = a.H_q * a.D / 8, pk = a.H_kv * a.D / 8;   // 16-byte pieces per token row
  for (int p = threadIdx.x; p < pq + pk; p += kPoolThreads) {
    const bool is_q = p < pq;
    const int pp = is_q ? p : p - pq;
    const int H = is_q ? a.H_q : a.H_kv;
    if (is_q && !a.heads.has(pp / (a.D / 8))) continue;   // a head of another pattern
    const uint16_t *src = static_cast<const uint16_t *>(is_q ? a.q : a.k) +
                          (static_cast<size_t>(b) * a.S + t0) * H * a.D + static_cast<size_t>(pp) * 8;
    const size_t stride = static_cast<size_t>(H) * a.D;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int r = 0;
    for (; r + 8 <= rows; r += 8) {
      uint4 u[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) u[x] = __ldg(reinterpret_cast<const uint4 *>(src + (r + x) * stride));
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const uint32_t w[4] = {u[x].x, u[x].y, u[x].z, u[x].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          acc[2 * c] += bf16_lo(w[c]);
          acc[2 * c + 1] += bf16_hi(w[c]);
        }
      }
    }
    for (; r < rows; ++r) {
      const uint4 u = __ldg(reinterpret_cast<const uint4 *>(src + r * stride));
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        acc[2 * c] += bf16_lo(w[c]);
        acc[2 * c + 1] += bf16_hi(w[c]);
      }
    }
    // q: [B, H_q, nb, D]; k: transposed [B, H_kv, D, nb]; debug copies [B, H, nb, D]
    const int h = pp / (a.D / 8), d0 = (pp - h * (a.D / 8)) * 8;
    const size_t o = ((static_cast<size_t>(b) * H + h) * a.nb + j) * a.D + d0;
    const float4 v0 = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    const float4 v1 = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
    if (is_q) {
      reinterpret_cast<float4 *>(a.q_pool + o)[0] = v0;
      reinterpret_cast<float4 *>(a.q_pool + o)[1] = v1;
    } else {
      float *kt = a.k_pool + (static_cast<size_t>(b) * H + h) * a.D * static_cast<size_t>(a.nb) + j;
#pragma unroll
      for (int x = 0; x < 8; ++x) kt[static_cast<size_t>(d0 + x) * a.nb] = acc[x] * inv;
    }
    float *dbg = is_q ? a.dbg_q_pool : a.dbg_k_pool;
    if (dbg) {
      reinterpret_cast<float4 *>(dbg + o)[0] = v0;
      reinterpret_cast<float4 *>(dbg + o)[1] = v1;
    }
  }
}

// ------------------------------------------------------------------------------ scores + top-k

constexpr int kTopThreads = 256;
constexpr int kKeysPerPass = 2 * kTopThreads;   // two key blocks per thread and pass

inline size_t bs_smem_bytes(int R, int nb, int D) {
  return (static_cast<size_t>(R) * D + static_cast<size_t>(R) * nb + 8 * 256) * 4;
}

// Top-k of s[0 .. n) (n > k) for one warp by an 8-bit radix select over the order-
// preserving keys: writes the kept indices ascending to out.  The general path (any
// values, many equal ones); warp_topk_bucket below is the usual one.
__device__ void warp_topk_radix(const float *s, int n, int k, int *hist, int32_t *out) {
  const int lane = threadIdx.x & 31;
  uint32_t prefix = 0u, mask = 0u;
  int need = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
    for (int j = lane; j < n; j += 32) {
      const uint32_t key = ordered_key(s[j]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncwarp();
    // bins from the top: lane l owns 255 - 8l .. 255 - 8l - 7
    int c[8], sum = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      c[u] = hist[255 - 8 * lane - u];
      sum += c[u];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    const int excl = incl - sum;
    const unsigned owner = __ballot_sync(kFull, excl < need && need <= incl);
    const int src = __ffs(owner) - 1;
    int bin = 0, above = 0;
    if (lane == src) {
      int acc = excl;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (acc + c[u] >= need) {
          bin = 255 - 8 * lane - u;
          above = acc;
          break;
        }
        acc += c[u];
      }
    }
    bin = __shfl_sync(kFull, bin, src);
    above = __shfl_sync(kFull, above, src);
    need -= above;
    prefix |= static_cast<uint32_t>(bin) << shift;
    mask |= 255u << shift;
    __syncwarp();
  }
  // keep every key above the threshold and the first `need` keys equal to it
  const uint32_t thr = prefix;
  const unsigned lt = (1u << lane) - 1u;
  int base = 0, eq_seen = 0;
  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    const uint32_t key = j < n ? ordered_key(s[j]) : 0u;
    const bool gt = j < n && key > thr;
    const bool eq = j < n && key == thr;
    const unsigned beq = __ballot_sync(kFull, eq);
    const bool take = gt || (eq && eq_seen + __popc(beq & lt) < need);
    const unsigned bt = __ballot_sync(kFull, take);
    if (take) out[base + __popc(bt & lt)] = j;
    base += __popc(bt);
    eq_seen += __popc(beq);
  }
}

// Top-k of s[0 .. n) (n > k) for one warp, ascending into out.  The scores are spread
// over 256 buckets by value between the row's min and max (a map that never decreases
// with the score, so a higher bucket holds only larger scores); one histogram and a
// scan from the top find the bucket holding the k-th largest score; that bucket's
// members (at most 32, else the radix select runs) are ranked exactly: larger score,
// then smaller index.  Kept members are marked in s (a NaN pattern no score has), and
// one pass writes every index above the bucket or marked.
__device__ void warp_topk_bucket(float *s, int n, int k, int *hist, int32_t *out) {
  const int lane = threadIdx.x & 31;
  float mn = INFINITY, mx = -INFINITY;
  for (int j = lane; j < n; j += 32) {
    mn = fminf(mn, s[j]);
    mx = fmaxf(mx, s[j]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(kFull, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
  }
  const unsigned lt = (1u << lane) - 1u;
  if (!(mx > mn)) {   // every score equal: the k smallest indices
    for (int j = lane; j < k; j += 32) out[j] = j;
    return;
  }
  const float sc = 256.f / (mx - mn);
  auto bucket = [&](float x) { return min(255, static_cast<int>((x - mn) * sc)); };
  for (int i = lane; i < 256; i += 32) hist[i] = 0;
  __syncwarp();
  for (int j = lane; j < n; j += 32) atomicAdd(&hist[bucket(s[j])], 1);
  __syncwarp();
  int c[8], sum = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    c[u] = hist[255 - 8 * lane - u];
    sum += c[u];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += v;
  }
  const int excl = incl - sum;
  const int src = __ffs(__ballot_sync(kFull, excl < k && k <= incl)) - 1;
  int bb = 0, above = 0, members = 0;
  if (lane == src) {
    int acc = excl;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (acc + c[u] >= k) {
        bb = 255 - 8 * lane - u;
        above = acc;
        members = c[u];
        break;
      }
      acc += c[u];
    }
  }
  bb = __shfl_sync(kFull, bb, src);
  above = __shfl_sync(kFull, above, src);
  members = __shfl_sync(kFull, members, src);
  const int need = k - above;   // members of bucket bb to keep, 1 .. members
  if (members > 32) {
    warp_topk_radix(s, n, k, hist, out);
    return;
  }
  // the bucket's members in index order (hist is free again): lane i takes member i
  __syncwarp();
  int got = 0;
  for (int j0 = 0; j0 < n && got < members; j0 += 32) {
    const int j = j0 + lane;
    const bool in = j < n && bucket(s[j]) == bb;
    const unsigned bal = __ballot_sync(kFull, in);
    if (in) hist[got + __popc(bal & lt)] = j;
    got += __popc(bal);
  }
  __syncwarp();
  const int my_j = lane < members ? hist[lane] : -1;
  const float my_s = my_j >= 0 ? s[my_j] : -INFINITY;
  int rank = 0;   // members ranked above this one
  for (int i = 0; i < members; ++i) {
    const int oj = __shfl_sync(kFull, my_j, i);
    const float os = __shfl_sync(kFull, my_s, i);
    rank += (os > my_s || (os == my_s && oj < my_j)) ? 1 : 0;
  }
  __syncwarp();
  if (my_j >= 0 && rank < need) s[my_j] = __uint_as_float(0xffffffffu);
  __syncwarp();
  int base = 0;
  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    bool take = false;
    if (j < n) {
      const float x = s[j];
      take = __float_as_uint(x) == 0xffffffffu || bucket(x) > bb;
    }
    const unsigned bt = __ballot_sync(kFull, take);
    if (take) out[base + __popc(bt & lt)] = j;
    base += __popc(bt);
  }
}

template <int D, int R>
__global__ void __launch_bounds__(kTopThreads) bs_topk_kernel(BsArgs a) {
  extern __shared__ __align__(16) float fsm[];
  float *s_q = fsm;                              // [R][D], pre-scaled
  float *s_sc = s_q + R * D;                     // [R][nb] scores
  int *s_hist = reinterpret_cast<int *>(s_sc + static_cast<size_t>(R) * a.nb);   // [8][256]
  const int tid = threadIdx.x, warp = tid >> 5;
  const int bh = blockIdx.y;                     // b * H_q + h
  const int b = bh / a.H_q, h = bh - b * a.H_q;
  if (!a.heads.has(h)) return;                   // a head of another pattern
  const int g = h / (a.H_q / a.H_kv);
  const int m0 = blockIdx.x * R;
  const int rows = min(R, a.nb - m0);
  const float *qp = a.q_pool + (static_cast<size_t>(bh) * a.nb + m0) * D;
  const float *kt = a.k_pool + (static_cast<size_t>(b) * a.H_kv + g) * D * static_cast<size_t>(a.nb);
  for (int e = tid; e < R * D; e += kTopThreads) s_q[e] = e < rows * D ? qp[e] * a.scale : 0.f;
  __syncthreads();
  const int n_keys = m0 + rows;                  // the last row's causal limit
  for (int kc = 0; kc < n_keys; kc += kKeysPerPass) {
    const int j0 = kc + tid, j1 = j0 + kTopThreads;
    const bool v0 = j0 < n_keys, v1 = j1 < n_keys;
    if (!v0) break;                              // j1 > j0: nothing left for this thread
    float acc0[R], acc1[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc0[r] = acc1[r] = 0.f;
#pragma unroll 4
    for (int d = 0; d < D; d += 4) {
      float k0[4], k1[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        k0[x] = kt[static_cast<size_t>(d + x) * a.nb + j0];
        k1[x] = v1 ? kt[static_cast<size_t>(d + x) * a.nb + j1] : 0.f;
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float4 qv = *reinterpret_cast<const float4 *>(s_q + r * D + d);
        acc0[r] = fmaf(qv.x, k0[0], fmaf(qv.y, k0[1], fmaf(qv.z, k0[2], fmaf(qv.w, k0[3], acc0[r]))));
        acc1[r] = fmaf(qv.x, k1[0], fmaf(qv.y, k1[1], fmaf(qv.z, k1[2], fmaf(qv.w, k1[3], acc1[r]))));
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r < rows) {
        s_sc[static_cast<size_t>(r) * a.nb + j0] = acc0[r];
        if (v1) s_sc[static_cast<size_t>(r) * a.nb + j1] = acc1[r];
      }
    }
  }
  __syncthreads();
  // one warp per row: row m keeps min(k_b, m + 1) of its m + 1 unmasked blocks
  for (int r = warp; r < rows; r += kTopThreads / 32) {
    const int m = m0 + r;
    const int n = m + 1;
    float *sr = s_sc + static_cast<size_t>(r) * a.nb;
    const size_t row = static_cast<size_t>(bh) * a.nb + m;
    int32_t *out = a.blk_idx + row * a.max_blk;
    const int lane = tid & 31;
    if (a.dbg_scores)
      for (int j = lane; j < n; j += 32) a.dbg_scores[row * a.nb + j] = sr[j];
    const int cnt = min(a.k_b, n);
    if (cnt == n) {
      for (int j = lane; j < n; j += 32) out[j] = j;
    } else if (cnt > 0) {
      warp_topk_bucket(sr, n, cnt, s_hist + warp * 256, out);
    }
    if (lane == 0) {
      a.blk_cnt[row] = cnt;
      a.col_cnt[row] = 0;
    }
  }
}

}  // namespace

cudaError_t launch_ashape(const AshapeArgs &a, cudaStream_t s) {
  dim3 grid((a.n_qblk + 7) / 8, a.BH);
  ProfScope ps("ashape_index", s);
  ashape_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

int bs_rows_per_cta(int nb, int D) {
  for (int R = 8; R >= 1; R >>= 1)   // prefer two CTAs per SM, then one
    if (bs_smem_bytes(R, nb, D) <= 100 * 1024) return R;
  for (int R = 8; R >= 1; R >>= 1)
    if (bs_smem_bytes(R, nb, D) <= 200 * 1024) return R;
  return 0;
}

cudaError_t launch_block_sparse(const BsArgs &a, cudaStream_t s) {
  cudaError_t e;
  {
    ProfScope ps("bs_pool", s);
    bs_pool_kernel<<<dim3(a.nb, a.B), kPoolThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int R = bs_rows_per_cta(a.nb, a.D);
  if (R < 1) return cudaErrorInvalidValue;
  const dim3 grid((a.nb + R - 1) / R, a.B * a.H_q);
  const size_t smem = bs_smem_bytes(R, a.nb, a.D);
  auto go = [&](auto kern) {
    cudaError_t st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (st != cudaSuccess) return st;
    ProfScope ps("bs_score_topk", s);
    kern<<<grid, kTopThreads, smem, s>>>(a);
    return cudaGetLastError();
  };
  auto pick = [&](auto dc) {
    constexpr int DD = decltype(dc)::value;
    switch (R) {
      case 8: return go(bs_topk_kernel<DD, 8>);
      case 4: return go(bs_topk_kernel<DD, 4>);
      case 2: return go(bs_topk_kernel<DD, 2>);
      default: return go(bs_topk_kernel<DD, 1>);
    }
  };
  return a.D == 128 ? pick(std::integral_constant<int, 128>{}) : pick(std::integral_constant<int, 64>{});
}

}  // namespace dsa
