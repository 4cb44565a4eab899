// Sparse causal prefill attention, warp-MMA (mma.sync) version.
//
// Source: "MInference 1.0: Accelerating Pre-filling for Long-Context LLMs via Dynamic
// Sparse Attention" (paper-graph-ui summary): "Vertical-Slash Hybrid Kernel" (Alg. 5:
// block phase over 64x64 tiles, then a column phase that gathers up to 64 listed key
// columns into a dense tile, one online softmax across both) and "Block-Sparse
// FlashAttention Kernel (Appendix C.4.1)"; masked attention of section 3.4 Eq. 1 with
// the mask constant taken as exact exclusion.
//
// One CTA (4 warps, 16 query rows each) per (query block m, query head h, batch b);
// query blocks are issued last-first because later blocks list more tiles.  K and V
// tiles (64 keys x D) are double-buffered in shared memory with 16-byte cp.async; a
// block tile is 64 consecutive keys, a column tile is 64 gathered key rows.  This is
// the portable baseline of the tensor-core prefill; see prefill_tc.cu for tcgen05.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "mma_sync.cuh"
#include "profile.h"

namespace dsa {
namespace {

constexpr int kPT = 64;   // keys per tile and rows per query block
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct PfSmem {
  static constexpr int kRow = D + 8;   // padded bf16 row (16 bytes of pad)
  static constexpr size_t kTileElems = static_cast<size_t>(kPT) * kRow;
  static constexpr size_t bytes() { return 4 * kTileElems * 2 + 2 * kPT * 4; }
};

template <int D>
__global__ void __launch_bounds__(128) prefill_mma_kernel(PrefillArgs a) {
  using SM = PfSmem<D>;
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t *s_k = reinterpret_cast<uint16_t *>(smem);           // [2][64][kRow]
  uint16_t *s_v = s_k + 2 * SM::kTileElems;                      // [2][64][kRow]
  int *s_pos = reinterpret_cast<int *>(s_v + 2 * SM::kTileElems);   // [2][64]

  const int S = a.S, n_qblk = (S + kPT - 1) / kPT;
  const int m = n_qblk - 1 - blockIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  const int G = a.H_q / a.H_kv, g = h / G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;
  const size_t bh = static_cast<size_t>(b) * a.H_q + h;
  const size_t list = bh * n_qblk + m;
  const int blk_cnt = min(max(a.blk_cnt[list], 0), a.max_blk);
  const int col_cnt = min(max(a.col_cnt[list], 0), a.max_col);
  const int32_t *bl = a.blk_idx + list * a.max_blk;
  const int32_t *cl = a.col_idx + list * a.max_col;
  const int n_tiles = blk_cnt + (col_cnt + kPT - 1) / kPT;
  const int last_row = m * kPT + kPT - 1;

  const uint16_t *kg = static_cast<const uint16_t *>(a.k) + (static_cast<size_t>(b) * S * a.H_kv + g) * D;
  const uint16_t *vg = static_cast<const uint16_t *>(a.v) + (static_cast<size_t>(b) * S * a.H_kv + g) * D;
  const size_t krow = static_cast<size_t>(a.H_kv) * D;

  auto tile_pos = [&](int t, int x) -> int {
    if (t < blk_cnt) {
      const int n = bl[t];
      if (n < 0 || n > m) return -1;
      const int j = n * kPT + x;
      return j < S ? j : -1;
    }
    const int c = (t - blk_cnt) * kPT + x;
    if (c >= col_cnt) return -1;
    const int j = cl[c];
    return (j >= 0 && j < S && j <= last_row) ? j : -1;
  };
  auto load_tile = [&](int t, int buf) {
    constexpr int CH = D * 2 / 16;
    uint16_t *dk = s_k + buf * SM::kTileElems;
    uint16_t *dv = s_v + buf * SM::kTileElems;
    if (tid < kPT) s_pos[buf * kPT + tid] = tile_pos(t, tid);
    for (int e = tid; e < kPT * CH; e += 128) {
      const int key = e / CH, c = e - key * CH;
      const int j = tile_pos(t, key);
      uint16_t *pk = dk + key * SM::kRow + c * 8;
      uint16_t *pv = dv + key * SM::kRow + c * 8;
      if (j >= 0) {
        cp_async_16(pk, kg + static_cast<size_t>(j) * krow + c * 8);
        cp_async_16(pv, vg + static_cast<size_t>(j) * krow + c * 8);
      } else {
        *reinterpret_cast<uint4 *>(pk) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(pv) = make_uint4(0, 0, 0, 0);
      }
    }
  };

  // Q fragments of this warp's 16 rows
  const int r_lo = m * kPT + warp * 16 + gq, r_hi = r_lo + 8;
  uint32_t qa[D / 16][4];
  {
    const uint16_t *qg = static_cast<const uint16_t *>(a.q);
    const uint32_t *q_lo = reinterpret_cast<const uint32_t *>(
        qg + ((static_cast<size_t>(b) * S + min(r_lo, S - 1)) * a.H_q + h) * D);
    const uint32_t *q_hi = reinterpret_cast<const uint32_t *>(
        qg + ((static_cast<size_t>(b) * S + min(r_hi, S - 1)) * a.H_q + h) * D);
#pragma unroll
    for (int kb = 0; kb < D / 16; ++kb) {
      qa[kb][0] = r_lo < S ? q_lo[kb * 8 + tq] : 0u;
      qa[kb][1] = r_hi < S ? q_hi[kb * 8 + tq] : 0u;
      qa[kb][2] = r_lo < S ? q_lo[kb * 8 + 4 + tq] : 0u;
      qa[kb][3] = r_hi < S ? q_hi[kb * 8 + 4 + tq] : 0u;
    }
  }
  float o[D / 8][4];
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[nd][c] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  const float sl2 = a.scale * kLog2e;

  if (n_tiles > 0) {
    load_tile(0, 0);
    cp_async_commit();
  }
  for (int t = 0; t < n_tiles; ++t) {
    const int buf = t & 1;
    if (t + 1 < n_tiles) {
      load_tile(t + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint16_t *Ks = s_k + buf * SM::kTileElems;
    const uint16_t *Vs = s_v + buf * SM::kTileElems;
    const int *pos = s_pos + buf * kPT;
    const int mi = lane >> 3, ri = lane & 7;
    float sc[8][4];
#pragma unroll
    for (int nb = 0; nb < 8; ++nb)
#pragma unroll
      for (int c = 0; c < 4; ++c) sc[nb][c] = 0.f;
#pragma unroll
    for (int kb = 0; kb < D / 16; ++kb) {
#pragma unroll
      for (int nb2 = 0; nb2 < 4; ++nb2) {
        uint32_t r[4];
        ldsm_x4(r, Ks + (nb2 * 16 + (mi >> 1) * 8 + ri) * SM::kRow + kb * 16 + (mi & 1) * 8);
        mma_16816(sc[2 * nb2], qa[kb], r[0], r[1]);
        mma_16816(sc[2 * nb2 + 1], qa[kb], r[2], r[3]);
      }
    }
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 8; ++nb)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int j = pos[nb * 8 + 2 * tq + c];
        sc[nb][c] = (j >= 0 && j <= r_lo) ? sc[nb][c] * sl2 : -INFINITY;
        sc[nb][2 + c] = (j >= 0 && j <= r_hi) ? sc[nb][2 + c] * sl2 : -INFINITY;
        mx_lo = fmaxf(mx_lo, sc[nb][c]);
        mx_hi = fmaxf(mx_hi, sc[nb][2 + c]);
      }
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(kFull, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(kFull, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(kFull, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(kFull, mx_hi, 2));
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float al_lo = mn_lo == -INFINITY ? 1.f : fast_exp2(m_lo - mn_lo);
    const float al_hi = mn_hi == -INFINITY ? 1.f : fast_exp2(m_hi - mn_hi);
    float ps_lo = 0.f, ps_hi = 0.f;
#pragma unroll
    for (int nb = 0; nb < 8; ++nb)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const float p0 = mn_lo == -INFINITY ? 0.f : fast_exp2(sc[nb][c] - mn_lo);
        const float p1 = mn_hi == -INFINITY ? 0.f : fast_exp2(sc[nb][2 + c] - mn_hi);
        sc[nb][c] = p0;
        sc[nb][2 + c] = p1;
        ps_lo += p0;
        ps_hi += p1;
      }
    l_lo = l_lo * al_lo + ps_lo;
    l_hi = l_hi * al_hi + ps_hi;
    m_lo = mn_lo;
    m_hi = mn_hi;
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      o[nd][0] *= al_lo;
      o[nd][1] *= al_lo;
      o[nd][2] *= al_hi;
      o[nd][3] *= al_hi;
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16x2(sc[2 * kk][0], sc[2 * kk][1]);
      pa[1] = pack_bf16x2(sc[2 * kk][2], sc[2 * kk][3]);
      pa[2] = pack_bf16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      pa[3] = pack_bf16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
      for (int nd2 = 0; nd2 < D / 16; ++nd2) {
        uint32_t r[4];
        ldsm_x4_trans(r, Vs + (kk * 16 + (mi & 1) * 8 + ri) * SM::kRow + nd2 * 16 + (mi >> 1) * 8);
        mma_16816(o[2 * nd2], pa, r[0], r[1]);
        mma_16816(o[2 * nd2 + 1], pa, r[2], r[3]);
      }
    }
    __syncthreads();
  }
  l_lo += __shfl_xor_sync(kFull, l_lo, 1);
  l_lo += __shfl_xor_sync(kFull, l_lo, 2);
  l_hi += __shfl_xor_sync(kFull, l_hi, 1);
  l_hi += __shfl_xor_sync(kFull, l_hi, 2);
  const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f;
  const float inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
  uint16_t *og = static_cast<uint16_t *>(a.out);
  if (r_lo < S) {
    uint32_t *orow = reinterpret_cast<uint32_t *>(og + ((static_cast<size_t>(b) * S + r_lo) * a.H_q + h) * D);
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) orow[nd * 4 + tq] = pack_bf16x2(o[nd][0] * inv_lo, o[nd][1] * inv_lo);
    if (a.lse && tq == 0) a.lse[bh * S + r_lo] = l_lo > 0.f ? (m_lo + log2f(l_lo)) * kLn2 : -INFINITY;
  }
  if (r_hi < S) {
    uint32_t *orow = reinterpret_cast<uint32_t *>(og + ((static_cast<size_t>(b) * S + r_hi) * a.H_q + h) * D);
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) orow[nd * 4 + tq] = pack_bf16x2(o[nd][2] * inv_hi, o[nd][3] * inv_hi);
    if (a.lse && tq == 0) a.lse[bh * S + r_hi] = l_hi > 0.f ? (m_hi + log2f(l_hi)) * kLn2 : -INFINITY;
  }
}

template <int D>
cudaError_t launch_prefill_mma_d(const PrefillArgs &a, cudaStream_t s) {
  const size_t smem = PfSmem<D>::bytes();
  auto kern = prefill_mma_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.S + kPT - 1) / kPT, a.H_q, a.B);
  {
    ProfScope ps("prefill_attention_mma", s);
    kern<<<grid, 128, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_mma(const PrefillArgs &a, cudaStream_t s) {
  return a.D == 128 ? launch_prefill_mma_d<128>(a, s) : launch_prefill_mma_d<64>(a, s);
}

}  // namespace dsa
