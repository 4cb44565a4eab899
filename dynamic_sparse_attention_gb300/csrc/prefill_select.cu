// InfiniteHiP sparse prefill: the pruning stages for query blocks of 64 rows.
//
// Source: "InfiniteHiP: Extending Language Model Context Up to 3 Million Tokens on a
// Single GPU" (paper-graph-ui summary), section 3.4 "Formal Mechanism of a Single
// Pruning Stage" (Alg. 2: query blocks of b_q = 64 rows share one mask; the chunk
// score is the max over every head and every row of the block), "The Representative
// Token Selection Algorithm (SelectRep)" (Alg. 3) and "Prefill Latency Details"
// (chunked sparse prefill): query block m prunes the keys before its end.
//
// Every (query block, head, chunk) runs its own SelectRep tournament, and a probe is
// now a 64-row product: q_t . k for the block's 64 rows, of which the max decides.
// That is a dense contraction, so it runs on the tensor cores (mma.sync m16n8k16,
// bf16 in, fp32 out):
//  * one CTA per (query block, 64 chunks, KV head g); the H_kv CTAs of a query block
//    and chunk range form a thread-block cluster;
//  * warp w holds 16 rows of the block for query head g*G + w/4 as resident A
//    fragments (the 64 rows of a head are four warps);
//  * each tournament step gathers, with 16-byte cp.async, the probe row of every
//    (head, chunk) of the CTA -- G x 64 rows of 2*D bytes for KV head g -- into an
//    XOR-swizzled shared tile (the first two steps probe the same token for every head
//    of a chunk -- its first token, then its midpoint -- and gather one row per chunk
//    for all of them); each warp then scores its 16 rows against its head's 64 probes
//    (eight n-tiles), takes the max over its rows, and the four warps of a head
//    combine their maxima in shared memory; one thread per (head, chunk) moves the
//    tournament on;
//  * the chunk score (max over the group's heads) of the H_kv CTAs is combined in
//    distributed shared memory and written once.
// Rows past the sequence end take no part (their scores are -inf).
#include <cooperative_groups.h>
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "mma_sync.cuh"
#include "profile.h"

namespace dsa {
namespace {

constexpr int kCG = 64;    // chunks per CTA
constexpr int kBq = 64;    // query rows per block

template <int D, int G>
struct PfSmem {
  static constexpr int kRows = G * kCG;                      // probe rows per step
  static constexpr size_t kK = static_cast<size_t>(kRows) * D * 2;
  static constexpr size_t kRed = static_cast<size_t>(4) * kRows * 4;
  static constexpr size_t kState = static_cast<size_t>(kRows) * 4 * 4;   // lo, hi, best, x
  static size_t bytes(int L, bool explicit_list) {
    return kK + kRed + kState + kCG * 4 + (explicit_list ? static_cast<size_t>(kCG) * L * 4 : 0);
  }
};

__device__ __forceinline__ void cp16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(dst)), "l"(src));
}

template <int D>
__device__ __forceinline__ int swz(int row, int piece) {   // element offset, 8 bf16 per piece
  return row * D + ((piece ^ (row & 7)) << 3);
}

// two CTAs per SM (up to G = 4): the tournaments of both are in flight at once
template <int D, int G>
__global__ void __launch_bounds__(G * 4 * 32, G <= 4 ? 2 : 1) prefill_score_kernel(PfScoreArgs a) {
  namespace cg = cooperative_groups;
  using SM = PfSmem<D, G>;
  constexpr int NT = G * 4 * 32;
  constexpr int KS = D / 16;
  constexpr int PIECES = D / 8;
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t *s_k = reinterpret_cast<uint16_t *>(smem);
  float *s_red = reinterpret_cast<float *>(smem + SM::kK);                  // [4][G*kCG]
  int *s_lo = reinterpret_cast<int *>(smem + SM::kK + SM::kRed);           // [G*kCG]
  int *s_hi = s_lo + SM::kRows;
  float *s_best = reinterpret_cast<float *>(s_hi + SM::kRows);
  int *s_x = reinterpret_cast<int *>(s_best + SM::kRows);                  // probe this step, -1 none
  float *s_cmax = reinterpret_cast<float *>(s_x + SM::kRows);              // [kCG]
  int *s_pos = reinterpret_cast<int *>(s_cmax + kCG);                      // [kCG][L]

  grid_dep_wait();
  cg::cluster_group cluster = cg::this_cluster();
  const int g = static_cast<int>(cluster.block_rank());   // KV head (cluster along y)
  const int r = blockIdx.z;                                // query-block row: b * n_qblk + m
  const int b = r / a.n_qblk, m = r - b * a.n_qblk;
  const int c0 = blockIdx.x * kCG;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;

  // this row's input range (the same for every CTA of the cluster)
  int n_in, start = 0;
  const int32_t *in = nullptr;
  if (a.in_idx == nullptr) {
    const int Tm = min(max(a.kv_rows[r], 0), a.S);
    start = a.n_sink;
    n_in = max(0, Tm - a.n_stream - a.n_sink);
  } else {
    n_in = min(max(a.in_cnt[r], 0), a.in_stride);
    in = a.in_idx + static_cast<size_t>(r) * a.in_stride;
  }
  const int n_chunk = (n_in + a.L - 1) / a.L;
  if (c0 >= n_chunk) return;   // uniform across the cluster

  // positions of explicit lists, clamped to the key rows
  if (in) {
    for (int x = tid; x < kCG * a.L; x += NT) {
      const int c = x / a.L, o = x - c * a.L;
      const int e = (c0 + c) * a.L + o;
      s_pos[x] = e < n_in ? min(max(in[e], 0), a.S - 1) : 0;
    }
  }
  for (int i = tid; i < SM::kRows; i += NT) {
    const int c = i % kCG;
    const int len = c0 + c < n_chunk ? min(a.L, n_in - (c0 + c) * a.L) : 0;
    s_lo[i] = 0;
    s_hi[i] = len - 1;   // -1: no chunk
    s_best[i] = -INFINITY;
  }
  // the warp's 16 query rows of its head as A fragments
  const int hq = warp >> 2, mt = warp & 3;
  const int h = g * G + hq;
  const int row0 = kBq * m + 16 * mt + gq, row1 = row0 + 8;
  const bool ok0 = row0 < a.S, ok1 = row1 < a.S;
  uint32_t qa[KS][4];
  {
    const uint16_t *qb = static_cast<const uint16_t *>(a.q) + (static_cast<size_t>(b) * a.S) * a.H_q * D;
    auto qpair = [&](int row, bool ok, int d) -> uint32_t {
      if (!ok) return 0u;
      return *reinterpret_cast<const uint32_t *>(qb + (static_cast<size_t>(row) * a.H_q + h) * D + d);
    };
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = qpair(row0, ok0, ks * 16 + 2 * tq);
      qa[ks][1] = qpair(row1, ok1, ks * 16 + 2 * tq);
      qa[ks][2] = qpair(row0, ok0, ks * 16 + 8 + 2 * tq);
      qa[ks][3] = qpair(row1, ok1, ks * 16 + 8 + 2 * tq);
    }
  }
  const uint16_t *kg = static_cast<const uint16_t *>(a.k) + (static_cast<size_t>(b) * a.S * a.H_kv + g) * D;
  const size_t kstride = static_cast<size_t>(a.H_kv) * D;
  auto pos_of = [&](int c, int x) -> int { return in ? s_pos[c * a.L + x] : start + (c0 + c) * a.L + x; };
  __syncthreads();

  for (int step = 0;; ++step) {
    // this step's probe of every (head, chunk): the first token, then the midpoint
    int any = 0;
    for (int i = tid; i < SM::kRows; i += NT) {
      const int lo = s_lo[i], hi = s_hi[i];
      int x = -1;
      if (hi >= 0) {
        if (step == 0) x = 0;
        else if (lo < hi) x = (lo + hi + 1) >> 1;
      }
      s_x[i] = x;
      any |= x >= 0;
    }
    if (!__syncthreads_or(any)) break;
    // gather the probe rows (a row without a probe keeps what it held: its scores are
    // never read); the first two steps probe one token per chunk for every head
    const bool shared = step <= 1;
    const int n_rows = shared ? kCG : SM::kRows;
    for (int e = tid; e < n_rows * PIECES; e += NT) {
      const int i = e / PIECES, p = e - i * PIECES;
      const int x = s_x[i];
      if (x >= 0) cp16(s_k + swz<D>(i, p), kg + static_cast<size_t>(pos_of(i % kCG, x)) * kstride + p * 8);
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();
    // scores of the warp's 16 rows against its head's kCG probes; max over the rows
    {
      const int mtx = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int np = 0; np < kCG / 16; ++np) {   // pairs of n-tiles: 16 probes
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int krow = (shared ? 0 : hq * kCG) + np * 16 + (mtx >> 1) * 8 + rr;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t bk[4];
          ldsm_x4(bk, s_k + swz<D>(krow, 2 * ks + (mtx & 1)));
          mma_16816(acc[0], qa[ks], bk[0], bk[1]);
          mma_16816(acc[1], qa[ks], bk[2], bk[3]);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          float v0 = fmaxf(ok0 ? acc[nt][0] : -INFINITY, ok1 ? acc[nt][2] : -INFINITY);   // column 2tq
          float v1 = fmaxf(ok0 ? acc[nt][1] : -INFINITY, ok1 ? acc[nt][3] : -INFINITY);   // column 2tq+1
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            v0 = fmaxf(v0, __shfl_xor_sync(kFull, v0, o));
            v1 = fmaxf(v1, __shfl_xor_sync(kFull, v1, o));
          }
          if (gq == 0) {
            const int c = np * 16 + nt * 8 + 2 * tq;
            s_red[mt * SM::kRows + hq * kCG + c] = v0;
            s_red[mt * SM::kRows + hq * kCG + c + 1] = v1;
          }
        }
      }
    }
    __syncthreads();
    // move every tournament on: the right half wins only on a strictly higher score
    for (int i = tid; i < SM::kRows; i += NT) {
      const int x = s_x[i];
      if (x < 0) continue;
      const float sc = fmaxf(fmaxf(s_red[i], s_red[SM::kRows + i]),
                             fmaxf(s_red[2 * SM::kRows + i], s_red[3 * SM::kRows + i]));
      if (step == 0) {
        s_best[i] = sc;
      } else if (sc > s_best[i]) {
        s_lo[i] = x;
        s_best[i] = sc;
      } else {
        s_hi[i] = x - 1;
      }
    }
    __syncthreads();
  }
  // chunk maxima over this group's heads; representatives for inspection
  for (int c = tid; c < kCG; c += NT) {
    float mx = -INFINITY;
    for (int q = 0; q < G; ++q) mx = fmaxf(mx, s_best[q * kCG + c]);
    s_cmax[c] = mx;
  }
  if (a.dbg_rep) {
    for (int i = tid; i < SM::kRows; i += NT) {
      const int c = i % kCG, q = i / kCG;
      if (c0 + c < n_chunk) {
        const size_t o = (static_cast<size_t>(r) * a.H_q + g * G + q) * a.max_chunks + c0 + c;
        a.dbg_rep[o] = pos_of(c, s_lo[i]);
        if (a.dbg_rho) a.dbg_rho[o] = s_best[i];
      }
    }
  }
  cluster.sync();
  if (g == 0) {
    const int C = static_cast<int>(cluster.num_blocks());
    for (int c = tid; c < kCG; c += NT) {
      if (c0 + c >= n_chunk) continue;
      float mx = -INFINITY;
      for (int q = 0; q < C; ++q) mx = fmaxf(mx, *cluster.map_shared_rank(s_cmax + c, q));
      a.score[static_cast<size_t>(r) * a.max_chunks + c0 + c] = mx;
    }
  }
  cluster.sync();   // keep s_cmax until rank 0 has read it
}

// query block m sees the keys up to its last row
__global__ void prefill_rows_kernel(int32_t *kv_rows, int R, int n_qblk, int S) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r < R) kv_rows[r] = min(S, kBq * (r % n_qblk + 1));
}

// Query block m's attended set, sink U selection U window of T_m keys, in the tile /
// column form of the prefill kernel: the 64-key blocks lying wholly inside the sink or
// the window are tiles; every other attended key (the rest of the sink and the window,
// and the selected tokens) is a column, ascending.  The lists are shared by every head
// (the selection is the max over heads), so each row is written once per head.
__global__ void __launch_bounds__(128) prefill_lists_kernel(PfListArgs a) {
  const int r = blockIdx.x;
  const int b = r / a.n_qblk, m = r - b * a.n_qblk;
  const int Tm = min(a.S, kBq * (m + 1));
  const int ns = min(a.n_sink, Tm);
  const int ws = max(a.n_sink, Tm - a.n_stream);
  __shared__ int s_blk[512];
  __shared__ int s_nblk;
  auto full = [&](int j) {
    const int lo = kBq * j, hi = min(kBq * j + kBq, Tm);
    return ns >= ws || hi <= ns || lo >= ws;
  };
  if (threadIdx.x == 0) {
    int n = 0;
    const int j_sink = (ns + kBq - 1) / kBq;   // blocks touching the sink
    for (int j = 0; j < j_sink && n < 512; ++j)
      if (full(j)) s_blk[n++] = j;
    for (int j = max(j_sink, ws / kBq); j <= m && n < 512; ++j)
      if (full(j)) s_blk[n++] = j;
    s_nblk = n;
  }
  __syncthreads();
  const int nblk = min(s_nblk, a.max_blk);
  const int cnt = min(max(a.sel_cnt[r], 0), a.keep);
  const int32_t *sel = a.sel_idx + static_cast<size_t>(r) * a.keep;
  // columns: sink keys outside full blocks, the selection, window keys outside full blocks
  const int sink_cols = (ns >= ws || ns % kBq == 0) ? 0 : ns % kBq;   // the sink's partial last block
  const int w_lo = ws, w_hi = min(Tm, (ws + kBq - 1) / kBq * kBq);     // the window's partial first block
  const int win_cols = (ns >= ws || ws % kBq == 0) ? 0 : w_hi - w_lo;
  const int ncol = min(sink_cols + cnt + win_cols, a.max_col);
  for (int h = 0; h < a.H_q; ++h) {
    const size_t row = (static_cast<size_t>(b) * a.H_q + h) * a.n_qblk + m;
    int32_t *bl = a.blk_idx + row * a.max_blk;
    int32_t *cl = a.col_idx ? a.col_idx + row * a.max_col : nullptr;
    for (int i = threadIdx.x; i < nblk; i += blockDim.x) bl[i] = s_blk[i];
    if (cl) {
      for (int i = threadIdx.x; i < ncol; i += blockDim.x) {
        int v;
        if (i < sink_cols) v = ns - sink_cols + i;
        else if (i < sink_cols + cnt) v = sel[i - sink_cols];
        else v = w_lo + (i - sink_cols - cnt);
        cl[i] = v;
      }
    }
    if (threadIdx.x == 0) {
      a.blk_cnt[row] = nblk;
      a.col_cnt[row] = cl ? ncol : 0;
    }
  }
}

template <int D, int G>
cudaError_t launch_pf(const PfScoreArgs &a, cudaStream_t s) {
  const size_t smem = PfSmem<D, G>::bytes(a.L, a.in_idx != nullptr);
  auto kern = prefill_score_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // all of the unified L1 / shared memory as shared memory, so two CTAs fit an SM
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.max_chunks + kCG - 1) / kCG, a.H_kv, a.B * a.n_qblk);
  cfg.blockDim = dim3(G * 4 * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = a.H_kv;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

size_t prefill_score_smem(int D, int G, int L, bool explicit_list) {
  const size_t k = static_cast<size_t>(G) * kCG * D * 2;
  return k + static_cast<size_t>(4) * G * kCG * 4 + static_cast<size_t>(G) * kCG * 16 + kCG * 4 +
         (explicit_list ? static_cast<size_t>(kCG) * L * 4 : 0);
}

cudaError_t launch_prefill_lists(const PfListArgs &a, cudaStream_t s) {
  ProfScope ps("prefill_hip_lists", s);
  prefill_lists_kernel<<<a.B * a.n_qblk, 128, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_rows(int32_t *kv_rows, int R, int n_qblk, int S, cudaStream_t s) {
  prefill_rows_kernel<<<(R + 255) / 256, 256, 0, s>>>(kv_rows, R, n_qblk, S);
  return cudaGetLastError();
}

cudaError_t launch_prefill_score(const PfScoreArgs &a, cudaStream_t s) {
  if (a.max_chunks == 0) return cudaSuccess;
  const int G = a.H_q / a.H_kv;
  static const char *const kNames[4] = {"prefill_stage_score_s0", "prefill_stage_score_s1",
                                        "prefill_stage_score_s2", "prefill_stage_score_s3+"};
  ProfScope ps(kNames[a.stage < 3 ? a.stage : 3], s);
  if (a.D == 128) {
    switch (G) {
      case 1: return launch_pf<128, 1>(a, s);
      case 2: return launch_pf<128, 2>(a, s);
      case 4: return launch_pf<128, 4>(a, s);
      default: return launch_pf<128, 8>(a, s);
    }
  }
  switch (G) {
    case 1: return launch_pf<64, 1>(a, s);
    case 2: return launch_pf<64, 2>(a, s);
    case 4: return launch_pf<64, 4>(a, s);
    default: return launch_pf<64, 8>(a, s);
  }
}

}  // namespace dsa
