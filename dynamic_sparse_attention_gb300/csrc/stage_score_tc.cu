// InfiniteHiP pruning-stage scores with the SelectRep probes on the tensor cores.
//
// Source: "InfiniteHiP: Extending Language Model Context Up to 3 Million Tokens on a
// Single GPU" (paper-graph-ui summary), section 3.4: "The Representative Token
// Selection Algorithm (SelectRep)" (Alg. 3) and "Formal Mechanism of a Single Pruning
// Stage" (Alg. 2 steps 3-5).  The computation is that of stage_score_kernel in
// hip_select.cu (same tournament, same tie rule, same chunk score); only the way the
// probe dot products are formed differs.
//
// A probe of a tournament is the dot product of one key row with one query head.  One
// warp runs 16 tournaments at once -- 16 / G chunks times the G query heads of one KV
// group -- and forms each level's 16 probes with one 16 x 8 x D product on mma.sync:
// the 16 probed key rows are the A operand (row-major, straight from global memory into
// registers), the G query heads of the group the B operand (resident), so the scores
// of row R against every head of the group come out of the accumulators and the warp
// keeps the one of R's own head.  Against the scalar version (one 8-lane octet per
// tournament, three shuffles per probe) a lane holds four times the key bytes in flight
// and issues about a quarter of the instructions per probe.
//
// Operand layout.  In an m16n8k16 product, lane (quad g = lane / 4, t = lane % 4)
// supplies, for k-slice s, the elements 2t, 2t+1 (registers a0 / b0) and 2t+8, 2t+9
// (a2 / b1) of A rows g and g+8 and of B column g.  A dot product does not depend on
// the order of its terms, so the head dimension is permuted the same way for keys and
// queries: lane t reads the 16-byte pieces t, t+4, t+8, ... of a row (a quad reads 64
// contiguous bytes), and piece t + 4i feeds k-slices 2i (its words x, y) and 2i + 1
// (words z, w).
//
// One CTA = CPW = 16 / G chunks of one batch row, one warp per KV group; the chunk
// score (max over every query head) is formed in shared memory across the warps.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "mma_sync.cuh"

namespace dsa {

DSA_CHECK_WORD(stage_tc_check_word)

namespace {

constexpr int kTcMaxListSmem = 32 * 1024;   // bytes of staged list positions per CTA

template <int D, int G>
__global__ void __launch_bounds__(256, 4) stage_score_tc_kernel(StageScoreArgs a) {
  constexpr int NI = D / 32;      // 16-byte pieces of a row per lane
  constexpr int CPW = 16 / G;     // chunks per CTA (every warp covers all of them)
  extern __shared__ __align__(16) unsigned char smem[];
  float *s_rho = reinterpret_cast<float *>(smem);                  // [CPW][H_q]
  float *s_c0 = s_rho + CPW * a.H_q;                               // [warps][16][8] level-0 scores
  int *s_pos = reinterpret_cast<int *>(s_c0 + (blockDim.x >> 5) * 128);   // [CPW][L]

  grid_dep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, t = lane & 3;
  const int grp = warp;                    // KV group of this warp
  const int b = blockIdx.y, j0 = blockIdx.x * CPW;
  const size_t row_stride = static_cast<size_t>(a.H_kv) * D;
  const uint16_t *kb = static_cast<const uint16_t *>(a.k) + static_cast<size_t>(b) * a.T_max * row_stride +
                       static_cast<size_t>(grp) * D + 8 * t;
  const int32_t *lst = a.in_idx ? a.in_idx + static_cast<size_t>(b) * a.in_stride : nullptr;
  // explicit list: stage the CTA's positions (read before the count, which only bounds
  // what is used; a stale position is clamped to the key rows)
  if (lst) {
    const int n = CPW * a.L;
    for (int x = threadIdx.x; x < n; x += blockDim.x)
      s_pos[x] = min(max(__ldg(lst + min(j0 * a.L + x, a.in_stride - 1)), 0), a.T_max - 1);
  }
  // the group's query heads as B fragments (lane quad gq = head column gq)
  uint4 qf[NI];
  {
    const int h = grp * G + gq;
    if (gq < G) {
      const uint4 *qp = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.q) +
                                                        (static_cast<size_t>(b) * a.H_q + h) * D + 8 * t);
#pragma unroll
      for (int i = 0; i < NI; ++i) qf[i] = __ldg(qp + 4 * i);
    } else {
#pragma unroll
      for (int i = 0; i < NI; ++i) qf[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  int n_in, start;
  if (lst) {
    const int cnt_raw = a.in_cnt[b];
    DSA_CHECK(cnt_raw >= 0 && cnt_raw <= a.in_stride);
    n_in = min(max(cnt_raw, 0), a.in_stride);
    start = 0;
  } else {
    const int kv_raw = a.kv_len[b];
    DSA_CHECK(kv_raw >= 0 && kv_raw <= a.T_max);
    const int Tb = min(max(kv_raw, 0), a.T_max);
    n_in = max(0, Tb - a.n_stream - a.n_sink);
    start = a.n_sink;
  }
  const int n_chunk = (n_in + a.L - 1) / a.L;
  if (j0 >= n_chunk) return;   // nothing in flight yet that outlives the CTA
#if DSA_CHECKS
  if (lst)   // the list entries this CTA uses (cached lists: as stored)
    for (int x = threadIdx.x; x < CPW * a.L; x += blockDim.x)
      if (j0 * a.L + x < n_in) {
        const int raw = __ldg(lst + j0 * a.L + x);
        DSA_CHECK(raw >= 0 && raw < a.T_max);
      }
#endif
  __syncthreads();             // staged positions

  auto pos_of = [&](int c, int x) -> int {
    return lst ? s_pos[c * a.L + x] : min(start + (j0 + c) * a.L + x, a.T_max - 1);
  };
  auto len_of = [&](int c) -> int { return min(a.L, n_in - (j0 + c) * a.L); };   // <= 0: none
  // 16 x 8 x D product of the A rows held by this lane with the resident query heads
  auto product = [&](const uint4 *ra, const uint4 *rb, float *c) {
    c[0] = c[1] = c[2] = c[3] = 0.f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const uint32_t a_lo[4] = {ra[i].x, rb[i].x, ra[i].y, rb[i].y};
      mma_16816(c, a_lo, qf[i].x, qf[i].y);
      const uint32_t a_hi[4] = {ra[i].z, rb[i].z, ra[i].w, rb[i].w};
      mma_16816(c, a_hi, qf[i].z, qf[i].w);
    }
  };
  auto load_row = [&](uint4 *r, int pos, bool on) {
    if (on) {
      const uint4 *p = reinterpret_cast<const uint4 *>(kb + static_cast<size_t>(pos) * row_stride);
#pragma unroll
      for (int i = 0; i < NI; ++i) r[i] = __ldg(p + 4 * i);
    } else {
#pragma unroll
      for (int i = 0; i < NI; ++i) r[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  };

  // tournaments of this quad: R0 = gq and R1 = gq + 8 (chunk R / G, head R % G)
  const int hh = gq % G;
  const int cA = gq / G, cB = (gq + 8) / G;
  const int lenA = len_of(cA), lenB = len_of(cB);
  // level 0: rows 0 and the first midpoint of every chunk (shared by all G heads) are
  // the A rows 2c and 2c + 1
  {
    uint4 ra[NI], rb[NI];
    const int r0 = gq, r1 = gq + 8;
    const int c0 = r0 >> 1, c1 = r1 >> 1;
    const int l0 = c0 < CPW ? len_of(c0) : 0, l1 = c1 < CPW ? len_of(c1) : 0;
    const int x0 = (r0 & 1) ? (l0 >> 1) : 0, x1 = (r1 & 1) ? (l1 >> 1) : 0;
    const bool on0 = l0 > 0 && ((r0 & 1) == 0 || l0 > 1);
    const bool on1 = l1 > 0 && ((r1 & 1) == 0 || l1 > 1);
    load_row(ra, on0 ? pos_of(c0, x0) : 0, on0);
    load_row(rb, on1 ? pos_of(c1, x1) : 0, on1);
    float c[4];
    product(ra, rb, c);
    float *sc = s_c0 + warp * 128;
    sc[gq * 8 + 2 * t] = c[0];
    sc[gq * 8 + 2 * t + 1] = c[1];
    sc[(gq + 8) * 8 + 2 * t] = c[2];
    sc[(gq + 8) * 8 + 2 * t + 1] = c[3];
    __syncwarp();
  }
  const float *sc = s_c0 + warp * 128;
  int loA = 0, hiA = lenA - 1, loB = 0, hiB = lenB - 1;
  float sA = lenA > 0 ? sc[(2 * cA) * 8 + hh] : -INFINITY;
  float sB = lenB > 0 ? sc[(2 * cB) * 8 + hh] : -INFINITY;
  // the first halving (its right score is the level-0 midpoint row)
  if (loA < hiA) {
    const int mid = (loA + hiA + 1) >> 1;
    const float sm = sc[(2 * cA + 1) * 8 + hh];
    if (sm > sA) { loA = mid; sA = sm; } else { hiA = mid - 1; }
  }
  if (loB < hiB) {
    const int mid = (loB + hiB + 1) >> 1;
    const float sm = sc[(2 * cB + 1) * 8 + hh];
    if (sm > sB) { loB = mid; sB = sm; } else { hiB = mid - 1; }
  }
  // remaining levels: one probe per active tournament per product
  const int src = 4 * gq + (hh >> 1);
  while (__any_sync(kFull, loA < hiA || loB < hiB)) {
    const bool onA = loA < hiA, onB = loB < hiB;
    const int midA = (loA + hiA + 1) >> 1, midB = (loB + hiB + 1) >> 1;
    uint4 ra[NI], rb[NI];
    load_row(ra, onA ? pos_of(cA, midA) : 0, onA);
    load_row(rb, onB ? pos_of(cB, midB) : 0, onB);
    float c[4];
    product(ra, rb, c);
    const float vA = (hh & 1) ? c[1] : c[0];
    const float vB = (hh & 1) ? c[3] : c[2];
    const float smA = __shfl_sync(kFull, vA, src);
    const float smB = __shfl_sync(kFull, vB, src);
    if (onA) {
      if (smA > sA) { loA = midA; sA = smA; } else { hiA = midA - 1; }
    }
    if (onB) {
      if (smB > sB) { loB = midB; sB = smB; } else { hiB = midB - 1; }
    }
  }
  if (t == 0) {
    const int h = grp * G + hh;
    if (lenA > 0) {
      s_rho[cA * a.H_q + h] = sA;
      if (a.dbg_rep) {
        const size_t o = (static_cast<size_t>(b) * a.H_q + h) * a.max_chunks + j0 + cA;
        a.dbg_rep[o] = pos_of(cA, loA);
        if (a.dbg_rho) a.dbg_rho[o] = sA;
      }
    }
    if (lenB > 0) {
      s_rho[cB * a.H_q + h] = sB;
      if (a.dbg_rep) {
        const size_t o = (static_cast<size_t>(b) * a.H_q + h) * a.max_chunks + j0 + cB;
        a.dbg_rep[o] = pos_of(cB, loB);
        if (a.dbg_rho) a.dbg_rho[o] = sB;
      }
    }
  }
  __syncthreads();
  // chunk score: max over all query heads, one warp per chunk
  const int n_here = min(CPW, n_chunk - j0);
  for (int c = warp; c < n_here; c += blockDim.x >> 5) {
    float m = -INFINITY;
    for (int i = lane; i < a.H_q; i += 32) m = fmaxf(m, s_rho[c * a.H_q + i]);
    m = warp_max(m);
    if (lane == 0) a.score[static_cast<size_t>(b) * a.max_chunks + j0 + c] = m;
  }
}

size_t tc_smem(const StageScoreArgs &a, int cpw) {
  return static_cast<size_t>(cpw) * a.H_q * 4 + static_cast<size_t>(a.H_kv) * 128 * 4 +
         (a.in_idx ? static_cast<size_t>(cpw) * a.L * 4 : 0);
}

template <int D, int G>
cudaError_t launch_tc(const StageScoreArgs &a, cudaStream_t s) {
  constexpr int CPW = 16 / G;
  const size_t smem = tc_smem(a, CPW);
  auto kern = stage_score_tc_kernel<D, G>;
  if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 grid((a.max_chunks + CPW - 1) / CPW, a.B);
  launch_pdl(kern, grid, dim3(32 * a.H_kv), smem, s, a);
  return cudaGetLastError();
}

}  // namespace

bool stage_score_tc_ok(const StageScoreArgs &a) {
  if (a.dtype != DSA_BF16 || a.T_q != 1 || (a.D != 64 && a.D != 128)) return false;
  const int G = a.H_q / a.H_kv;
  if (G != 2 && G != 4 && G != 8) return false;
  // Measured on GB300 (1M, 128K and batch-16 workloads): short tournaments (chunks of
  // 4 and 16 tokens) are faster here, long ones (64 and 256) in the scalar kernel, whose
  // one-chunk CTAs keep more tournaments resident.
  if (a.H_kv > 8 || a.L < 2 || a.L > 16) return false;   // 256 threads at most (launch bounds)
  return !a.in_idx || static_cast<size_t>(16 / G) * a.L * 4 <= kTcMaxListSmem;
}

cudaError_t launch_stage_score_tc(const StageScoreArgs &a, cudaStream_t s) {
  if (a.max_chunks == 0) return cudaSuccess;
  const int G = a.H_q / a.H_kv;
  if (a.D == 128) {
    if (G == 2) return launch_tc<128, 2>(a, s);
    if (G == 4) return launch_tc<128, 4>(a, s);
    return launch_tc<128, 8>(a, s);
  }
  if (G == 2) return launch_tc<64, 2>(a, s);
  if (G == 4) return launch_tc<64, 4>(a, s);
  return launch_tc<64, 8>(a, s);
}

}  // namespace dsa
