// MInference vertical-slash index build on sm_103a.
//
// Source: "MInference 1.0: Accelerating Pre-filling for Long-Context LLMs via Dynamic
// Sparse Attention" (paper-graph-ui summary), section 3.4 "Online Dynamic Index
// Estimation: Vertical-Slash Heads" (Alg. 2 steps 1-4) and "Vertical-Slash Hybrid
// Kernel" (Alg. 4, the two-way merge into block and column lists).
//
// Kernels, in launch order:
//   vs_pass<0>   per (key split, KV head, batch): scores of the last r <= 64 queries of
//                the G query heads of this KV head against the split's 64-key tiles
//                (bf16 mma, fp32 accumulate), online row max / row sum partials;
//   vs_stats     combine the partials into the final row max and row sum;
//   vs_pass<1>   recompute the scores, normalise, and per 64-key tile write the column
//                sums (one tile -> one owner, no atomics) and per-tile diagonal sums
//                (127 offsets per tile), all in a fixed order -> deterministic;
//   vs_slash     add the <= 2 tile partials of every offset in ascending tile order;
//   vs_topk      per (batch, head, {vertical, slash}): radix select of the k largest
//                (ties -> smaller index) and an ascending compaction;
//   vs_convert   per (batch, head, run of query blocks): the slash offsets become a
//                bitmap of block diagonals d = m - n; block m lists n = m - d for every
//                d <= m, and keeps the vertical columns whose block is not listed.
// Scores are base-2 logits (scale * log2 e folded in); the probabilities are the same.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "mma_sync.cuh"
#include "profile.h"

namespace dsa {
namespace {

constexpr int kKT = kVsKeyTile;        // 64 keys per tile
constexpr int kRowsPerHead = 64;       // estimate rows per head slot (r = min(last_q, S) used)
constexpr int kDiag = kKT + kRowsPerHead - 1;   // 127 offsets touched by one tile
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct VsSmem {
  static constexpr int kRowK = D + 8;  // bf16 elements per padded K row (16-byte pad)
  static constexpr int kPRow = kKT + 4;  // floats per padded P row
  static size_t bytes(bool pass1) {
    size_t o = 2ull * kKT * kRowK * 2;                             // double-buffered K tiles
    if (pass1) {
      o += static_cast<size_t>(4) * kRowsPerHead * kPRow * 4;     // P tile per head slot
      o += static_cast<size_t>(8) * kKT * 4;                      // per-warp column partials
    }
    return o;
  }
};

struct VsPassArgs {
  VsArgs a;
  int G, r_q, n_split, tiles_per_split;
  int n_hgroups;   // CTAs per KV head along y: each serves up to kSlots query heads
};
constexpr int kSlots = 4;   // query heads per CTA (two warps each)

template <int D, int PASS>
__global__ void __launch_bounds__(64 * kSlots) vs_pass_kernel(VsPassArgs pa) {
  using SM = VsSmem<D>;
  const VsArgs &a = pa.a;
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t *s_k = reinterpret_cast<uint16_t *>(smem);
  float *s_P = reinterpret_cast<float *>(smem + 2ull * kKT * SM::kRowK * 2);
  float *s_col = s_P + static_cast<size_t>(kSlots) * kRowsPerHead * SM::kPRow;

  const int split = blockIdx.x, b = blockIdx.z;
  const int g = blockIdx.y / pa.n_hgroups;
  const int hs0 = (blockIdx.y % pa.n_hgroups) * kSlots;   // first head slot of this CTA
  const int n_slots = min(kSlots, pa.G - hs0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x;
  const int G = pa.G, S = a.S, r_q = pa.r_q;
  const int hs = hs0 + (warp >> 1);         // head slot inside the group
  const bool slot_ok = hs < G;              // warps past the group's last head stay idle
  const int h = g * G + (slot_ok ? hs : 0);
  const int row0 = (warp & 1) * 32;         // first of this warp's 32 estimate rows
  const int gq = lane >> 2, tq = lane & 3;
  const int t_begin = split * pa.tiles_per_split;
  const int t_end = min(a.n_ktile, t_begin + pa.tiles_per_split);   // empty split: neutral partials

  const uint16_t *qg = static_cast<const uint16_t *>(a.q);
  const uint16_t *kg = static_cast<const uint16_t *>(a.k) +
                       (static_cast<size_t>(b) * S * a.H_kv + g) * D;
  const size_t krow = static_cast<size_t>(a.H_kv) * D;
  const float sl2 = a.scale * kLog2e;

  // A fragments of this warp's 32 query rows (rows >= r_q are zero and masked later)
  uint32_t qa[2][D / 16][4];
#pragma unroll
  for (int mb = 0; mb < 2; ++mb) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int i = row0 + mb * 16 + gq + half * 8;
      const bool ok = slot_ok && i < r_q;
      const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
          qg + ((static_cast<size_t>(b) * S + (S - r_q + (ok ? i : 0))) * a.H_q + h) * D);
#pragma unroll
      for (int kb = 0; kb < D / 16; ++kb) {
        qa[mb][kb][half] = ok ? qrow[kb * 8 + tq] : 0u;
        qa[mb][kb][2 + half] = ok ? qrow[kb * 8 + 4 + tq] : 0u;
      }
    }
  }
  // per-lane row state for its 4 rows: (mb, half)
  float m_run[2][2], l_run[2][2];
#pragma unroll
  for (int mb = 0; mb < 2; ++mb)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int i = row0 + mb * 16 + gq + hf * 8;
      if (PASS == 0) {
        m_run[mb][hf] = -INFINITY;
        l_run[mb][hf] = 0.f;
      } else {
        const size_t o = (static_cast<size_t>(b) * a.H_q + h) * kRowsPerHead + i;
        m_run[mb][hf] = slot_ok ? a.row_m[o] : -INFINITY;
        const float l = slot_ok ? a.row_l[o] : 0.f;
        l_run[mb][hf] = l > 0.f ? 1.f / l : 0.f;   // PASS 1 keeps the reciprocal
      }
    }

  auto load_tile = [&](int t, int buf) {
    uint16_t *dst = s_k + static_cast<size_t>(buf) * kKT * SM::kRowK;
    constexpr int CH = D * 2 / 16;
    for (int e = tid; e < kKT * CH; e += nthreads) {
      const int key = e / CH, c = e - key * CH;
      const int j = t * kKT + key;
      uint16_t *d = dst + key * SM::kRowK + c * 8;
      if (j < S) cp_async_16(d, kg + static_cast<size_t>(j) * krow + c * 8);
      else *reinterpret_cast<uint4 *>(d) = make_uint4(0, 0, 0, 0);
    }
  };

  if (t_begin < t_end) {
    load_tile(t_begin, 0);
    cp_async_commit();
  }
  for (int t = t_begin; t < t_end; ++t) {
    const int buf = (t - t_begin) & 1;
    if (t + 1 < t_end) {
      load_tile(t + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint16_t *kt = s_k + static_cast<size_t>(buf) * kKT * SM::kRowK;
    float sc[2][8][4];
#pragma unroll
    for (int mb = 0; mb < 2; ++mb)
#pragma unroll
      for (int nb = 0; nb < 8; ++nb)
#pragma unroll
        for (int c = 0; c < 4; ++c) sc[mb][nb][c] = 0.f;
#pragma unroll
    for (int kb = 0; kb < D / 16; ++kb) {
#pragma unroll
      for (int nb2 = 0; nb2 < 4; ++nb2) {
        // matrices: (keys 16nb2..+7, dims 16kb..), (same keys, dims 16kb+8..),
        //           (keys 16nb2+8..+15, dims 16kb..), (same, dims 16kb+8..)
        const int mi = lane >> 3, ri = lane & 7;
        const int key = nb2 * 16 + (mi >> 1) * 8 + ri;
        const int dim = kb * 16 + (mi & 1) * 8;
        uint32_t r[4];
        ldsm_x4(r, kt + key * SM::kRowK + dim);
#pragma unroll
        for (int mb = 0; mb < 2; ++mb) {
          mma_16816(sc[mb][2 * nb2], qa[mb][kb], r[0], r[1]);
          mma_16816(sc[mb][2 * nb2 + 1], qa[mb][kb], r[2], r[3]);
        }
      }
    }
    // mask + base-2 logits
    const int j0 = t * kKT;
#pragma unroll
    for (int mb = 0; mb < 2; ++mb)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int i = row0 + mb * 16 + gq + hf * 8;
        const int p = S - r_q + i;
#pragma unroll
        for (int nb = 0; nb < 8; ++nb)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int j = j0 + nb * 8 + 2 * tq + c;
            float &x = sc[mb][nb][hf * 2 + c];
            x = (i < r_q && j <= p) ? x * sl2 : -INFINITY;
          }
      }
    if (PASS == 0) {
#pragma unroll
      for (int mb = 0; mb < 2; ++mb)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          float mx = -INFINITY;
#pragma unroll
          for (int nb = 0; nb < 8; ++nb)
            mx = fmaxf(mx, fmaxf(sc[mb][nb][hf * 2], sc[mb][nb][hf * 2 + 1]));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
          const float m_new = fmaxf(m_run[mb][hf], mx);
          if (m_new != -INFINITY) {
            float s = 0.f;
#pragma unroll
            for (int nb = 0; nb < 8; ++nb)
              s += exp2f(sc[mb][nb][hf * 2] - m_new) + exp2f(sc[mb][nb][hf * 2 + 1] - m_new);
            l_run[mb][hf] = l_run[mb][hf] * exp2f(m_run[mb][hf] - m_new) + s;
            m_run[mb][hf] = m_new;
          }
        }
    } else {
      // probabilities; column partials over this warp's 32 rows; P tile to smem
      float *P = s_P + static_cast<size_t>(warp >> 1) * kRowsPerHead * SM::kPRow;
#pragma unroll
      for (int nb = 0; nb < 8; ++nb) {
        float c0 = 0.f, c1 = 0.f;
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const float m = m_run[mb][hf], inv = l_run[mb][hf];
            const float p0 = m != -INFINITY ? exp2f(sc[mb][nb][hf * 2] - m) * inv : 0.f;
            const float p1 = m != -INFINITY ? exp2f(sc[mb][nb][hf * 2 + 1] - m) * inv : 0.f;
            const int i = row0 + mb * 16 + gq + hf * 8;
            *reinterpret_cast<float2 *>(P + i * SM::kPRow + nb * 8 + 2 * tq) = make_float2(p0, p1);
            c0 += p0;
            c1 += p1;
          }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          c0 += __shfl_xor_sync(kFull, c0, o);
          c1 += __shfl_xor_sync(kFull, c1, o);
        }
        if (gq == 0) {
          s_col[warp * kKT + nb * 8 + 2 * tq] = c0;
          s_col[warp * kKT + nb * 8 + 2 * tq + 1] = c1;
        }
      }
      __syncthreads();
      // vertical sums: the two warps of a head slot, fixed order
      for (int e = tid; e < n_slots * kKT; e += nthreads) {
        const int slot = e / kKT, col = e - slot * kKT;
        const int j = j0 + col;
        if (j < S)
          a.vsum[(static_cast<size_t>(b) * a.H_q + g * G + hs0 + slot) * S + j] =
              s_col[(2 * slot) * kKT + col] + s_col[(2 * slot + 1) * kKT + col];
      }
      // diagonal sums of the tile: u = i - jj + 63, i.e. jj = i + 63 - u
      for (int e = tid; e < n_slots * kDiag; e += nthreads) {
        const int slot = e / kDiag, u = e - slot * kDiag;
        const float *Ps = s_P + static_cast<size_t>(slot) * kRowsPerHead * SM::kPRow;
        const int i_lo = max(0, u - (kKT - 1)), i_hi = min(kRowsPerHead - 1, u);
        float s = 0.f;
        for (int i = i_lo; i <= i_hi; ++i) s += Ps[i * SM::kPRow + i + (kKT - 1) - u];
        a.slash_part[((static_cast<size_t>(b) * a.H_q + g * G + hs0 + slot) * a.n_ktile + t) * kDiag + u] = s;
      }
    }
    __syncthreads();
  }
  if (PASS == 0) {
    // row partials of this split: quad-reduce the lane sums (m is quad-uniform)
#pragma unroll
    for (int mb = 0; mb < 2; ++mb)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float l = l_run[mb][hf];
        l += __shfl_xor_sync(kFull, l, 1);
        l += __shfl_xor_sync(kFull, l, 2);
        if (tq == 0 && slot_ok) {
          const int i = row0 + mb * 16 + gq + hf * 8;
          const size_t o = ((static_cast<size_t>(b) * a.H_kv + g) * pa.n_split + split) *
                               (G * kRowsPerHead) + hs * kRowsPerHead + i;
          a.part_m[o] = m_run[mb][hf];
          a.part_l[o] = l;
        }
      }
  }
}

__global__ void vs_stats_kernel(VsArgs a, int G, int n_split) {
  // one thread per (b, h, row)
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  const int total = a.B * a.H_q * kRowsPerHead;
  if (idx >= total) return;
  const int i = idx % kRowsPerHead;
  const int h = (idx / kRowsPerHead) % a.H_q;
  const int b = idx / (kRowsPerHead * a.H_q);
  const int g = h / G, hs = h - g * G;
  const float *pm = a.part_m + (static_cast<size_t>(b) * a.H_kv + g) * n_split * (G * kRowsPerHead) +
                    hs * kRowsPerHead + i;
  const float *pl = a.part_l + (pm - a.part_m);
  const size_t stride = static_cast<size_t>(G) * kRowsPerHead;
  float M = -INFINITY;
  for (int s = 0; s < n_split; ++s) M = fmaxf(M, pm[s * stride]);
  float L = 0.f;
  if (M != -INFINITY)
    for (int s = 0; s < n_split; ++s) {
      const float m = pm[s * stride];
      if (m != -INFINITY) L += pl[s * stride] * exp2f(m - M);
    }
  a.row_m[idx] = M;
  a.row_l[idx] = L;
}

__global__ void vs_slash_kernel(VsArgs a, int r_q) {
  const int o = blockIdx.x * blockDim.x + threadIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  const int S = a.S;
  if (o >= S || !a.heads.has(h)) return;
  // tile t covers offsets [S - r_q - 64t - 63, S - r_q - 64t + 63]
  const int base = S - r_q - (kKT - 1) - o;        // = 64t - u  for a covering tile
  int t_lo = base > 0 ? (base + kKT - 1) / kKT : 0;
  const int top = S - r_q + (kRowsPerHead - 1) - o;   // = 64t + (126 - u)... upper bound
  int t_hi = top >= 0 ? top / kKT : -1;
  if (t_hi > a.n_ktile - 1) t_hi = a.n_ktile - 1;
  const float *sp = a.slash_part + (static_cast<size_t>(b) * a.H_q + h) * a.n_ktile * kDiag;
  float s = 0.f;
  for (int t = t_lo; t <= t_hi; ++t) {
    const int u = o - (S - r_q - kKT * t - (kKT - 1));
    if (u >= 0 && u < kDiag) s += sp[static_cast<size_t>(t) * kDiag + u];
  }
  a.ssum[(static_cast<size_t>(b) * a.H_q + h) * S + o] = s;
}

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

template <int D>
cudaError_t launch_vs_d(const VsArgs &a, cudaStream_t s) {
  const int G = a.H_q / a.H_kv;
  const int r_q = min(a.last_q, a.S);
  VsPassArgs pa;
  pa.a = a;
  pa.G = G;
  pa.r_q = r_q;
  vs_plan(a.B, a.H_kv, a.n_ktile, &pa.n_split, &pa.tiles_per_split);
  pa.n_hgroups = (G + kSlots - 1) / kSlots;
  const int threads = 64 * min(G, kSlots);   // two warps per head slot
  dim3 grid(pa.n_split, a.H_kv * pa.n_hgroups, a.B);
  cudaError_t e;
  {
    const size_t smem = VsSmem<D>::bytes(false);
    auto k0 = vs_pass_kernel<D, 0>;
    e = cudaFuncSetAttribute(k0, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ProfScope ps("vs_pass_rowstats", s);
    k0<<<grid, threads, smem, s>>>(pa);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    const int total = a.B * a.H_q * kRowsPerHead;
    ProfScope ps("vs_combine_rowstats", s);
    vs_stats_kernel<<<(total + 255) / 256, 256, 0, s>>>(a, G, pa.n_split);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    const size_t smem = VsSmem<D>::bytes(true);
    auto k1 = vs_pass_kernel<D, 1>;
    e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ProfScope ps("vs_pass_sums", s);
    k1<<<grid, threads, smem, s>>>(pa);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    dim3 g2((a.S + 255) / 256, a.H_q, a.B);
    ProfScope ps("vs_combine_slash", s);
    vs_slash_kernel<<<g2, 256, 0, s>>>(a, r_q);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
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

void vs_plan(int B, int H_kv, int n_ktile, int *n_split, int *tiles_per_split) {
  // about two CTAs per SM of a 152-SM part; every split gets at least one tile
  int target = (304 + B * H_kv - 1) / (B * H_kv);
  if (target > n_ktile) target = n_ktile;
  if (target < 1) target = 1;
  const int tps = (n_ktile + target - 1) / target;
  *tiles_per_split = tps;
  *n_split = (n_ktile + tps - 1) / tps;
}

cudaError_t launch_vs_index(const VsArgs &a, cudaStream_t s) {
  return a.D == 128 ? launch_vs_d<128>(a, s) : launch_vs_d<64>(a, s);
}

}  // namespace dsa
