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
//  * bs_topk_kernel: one CTA per (b, query head, R consecutive query blocks).  The
//    pooled key blocks stream through shared memory (transposed, 128 at a time); each
//    thread scores one key block against R/2 of the R pooled query rows with fp32 FMAs
//    and the rows' scores stay in shared memory.  Then one warp per row finds the
//    k_b-th largest score by an 8-bit radix select over order-preserving keys and
//    writes the kept blocks in ascending order (larger score first, ties -> smaller
//    block index).  Softmax is monotone along a row, so the kernel ranks the scaled
//    logits; the causal mask is the row length m + 1.
#include <math.h>

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
    // pooled layout [B, H, nb, D]
    const int h = pp / (a.D / 8), d0 = (pp - h * (a.D / 8)) * 8;
    const size_t o = ((static_cast<size_t>(b) * H + h) * a.nb + j) * a.D + d0;
    float *dst = (is_q ? a.q_pool : a.k_pool) + o;
    float *dbg = is_q ? a.dbg_q_pool : a.dbg_k_pool;
    const float4 v0 = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    const float4 v1 = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
    reinterpret_cast<float4 *>(dst)[0] = v0;
    reinterpret_cast<float4 *>(dst)[1] = v1;
    if (dbg) {
      reinterpret_cast<float4 *>(dbg + o)[0] = v0;
      reinterpret_cast<float4 *>(dbg + o)[1] = v1;
    }
  }
}

// ------------------------------------------------------------------------------ scores + top-k

constexpr int kTopThreads = 256;
constexpr int kKeyChunk = 128;   // pooled key blocks staged per round

template <int D>
struct BsSmem {
  static constexpr int kTStride = kKeyChunk + 1;   // transposed chunk row (padded)
  static size_t bytes(int R, int nb) {
    return (static_cast<size_t>(R) * D + static_cast<size_t>(D) * kTStride +
            static_cast<size_t>(R) * nb + 8 * 256) * 4;
  }
};

// Top-k of s[0 .. n) (n > k) for one warp: writes the kept indices ascending to out.
__device__ void warp_topk_ascending(const float *s, int n, int k, int *hist, int32_t *out) {
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

template <int D>
__global__ void __launch_bounds__(kTopThreads) bs_topk_kernel(BsArgs a, int R) {
  extern __shared__ __align__(16) float fsm[];
  constexpr int kT = BsSmem<D>::kTStride;
  float *s_q = fsm;                              // [R][D]
  float *s_kt = s_q + R * D;                     // [D][kT] pooled keys, transposed
  float *s_sc = s_kt + D * kT;                   // [R][nb] scores
  int *s_hist = reinterpret_cast<int *>(s_sc + static_cast<size_t>(R) * a.nb);   // [8][256]
  const int tid = threadIdx.x, warp = tid >> 5;
  const int bh = blockIdx.y;                     // b * H_q + h
  const int b = bh / a.H_q, h = bh - b * a.H_q;
  const int g = h / (a.H_q / a.H_kv);
  const int m0 = blockIdx.x * R;
  const int rows = min(R, a.nb - m0);
  const float *qp = a.q_pool + (static_cast<size_t>(bh) * a.nb + m0) * D;
  const float *kp = a.k_pool + (static_cast<size_t>(b) * a.H_kv + g) * a.nb * static_cast<size_t>(D);
  for (int e = tid; e < R * D; e += kTopThreads) s_q[e] = e < rows * D ? qp[e] * a.scale : 0.f;
  const int n_keys = m0 + rows;                  // the last row's causal limit
  const int jj = tid & (kKeyChunk - 1), rg = tid >> 7;   // key of the chunk, row group (0/1)
  const int rpt = (R + 1) / 2;                   // rows per thread: rg, rg + 2, ...
  for (int kc = 0; kc < n_keys; kc += kKeyChunk) {
    __syncthreads();   // previous chunk consumed (and s_q written on the first round)
    const int nk = min(kKeyChunk, n_keys - kc);
    for (int e = tid; e < nk * (D / 4); e += kTopThreads) {
      const int r = e / (D / 4), d4 = e - r * (D / 4);
      const float4 v = reinterpret_cast<const float4 *>(kp + static_cast<size_t>(kc + r) * D)[d4];
      s_kt[(4 * d4 + 0) * kT + r] = v.x;
      s_kt[(4 * d4 + 1) * kT + r] = v.y;
      s_kt[(4 * d4 + 2) * kT + r] = v.z;
      s_kt[(4 * d4 + 3) * kT + r] = v.w;
    }
    __syncthreads();
    if (jj < nk) {
      float acc[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[u] = 0.f;
      for (int d = 0; d < D; d += 4) {
        const float k0 = s_kt[(d + 0) * kT + jj], k1 = s_kt[(d + 1) * kT + jj];
        const float k2 = s_kt[(d + 2) * kT + jj], k3 = s_kt[(d + 3) * kT + jj];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (u < rpt) {
            const int r = rg + 2 * u;
            if (r < R) {
              const float4 qv = *reinterpret_cast<const float4 *>(s_q + r * D + d);
              acc[u] = fmaf(qv.x, k0, fmaf(qv.y, k1, fmaf(qv.z, k2, fmaf(qv.w, k3, acc[u]))));
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int r = rg + 2 * u;
        if (u < rpt && r < rows) s_sc[static_cast<size_t>(r) * a.nb + kc + jj] = acc[u];
      }
    }
  }
  __syncthreads();
  // one warp per row: row m keeps min(k_b, m + 1) of its m + 1 unmasked blocks
  for (int r = warp; r < rows; r += kTopThreads / 32) {
    const int m = m0 + r;
    const int n = m + 1;
    const float *sr = s_sc + static_cast<size_t>(r) * a.nb;
    const size_t row = static_cast<size_t>(bh) * a.nb + m;
    int32_t *out = a.blk_idx + row * a.max_blk;
    const int lane = tid & 31;
    if (a.dbg_scores)
      for (int j = lane; j < n; j += 32) a.dbg_scores[row * a.nb + j] = sr[j];
    const int cnt = min(a.k_b, n);
    if (cnt == n) {
      for (int j = lane; j < n; j += 32) out[j] = j;
    } else if (cnt > 0) {
      warp_topk_ascending(sr, n, cnt, s_hist + warp * 256, out);
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
  for (int R = 16; R >= 1; R >>= 1) {
    const size_t smem = D == 128 ? BsSmem<128>::bytes(R, nb) : BsSmem<64>::bytes(R, nb);
    if (smem <= 200 * 1024) return R;
  }
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
  auto go = [&](auto kern, size_t smem) {
    cudaError_t st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (st != cudaSuccess) return st;
    ProfScope ps("bs_score_topk", s);
    kern<<<grid, kTopThreads, smem, s>>>(a, R);
    return cudaGetLastError();
  };
  return a.D == 128 ? go(bs_topk_kernel<128>, BsSmem<128>::bytes(R, a.nb))
                    : go(bs_topk_kernel<64>, BsSmem<64>::bytes(R, a.nb));
}

}  // namespace dsa
