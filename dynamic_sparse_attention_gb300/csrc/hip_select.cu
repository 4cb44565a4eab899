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
// is already known; each iteration therefore loads exactly one new key row.  Chunks of
// at most four tokens are scored from shared memory instead: one CTA copies all key
// rows of a few chunks in one round and runs their tournaments there.
//
// Layout of the top-K kernel: the row's chunk scores in registers, a bucket select for
// the K-th score, a block scan for the ranks of the kept chunks; the token list is
// written by several CTAs of the row, each repeating the selection.
#include <math.h>

#include <algorithm>

#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "mma_sync.cuh"

namespace dsa {

DSA_CHECK_WORD(hip_select_check_word)

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
    const int kv_raw = kv_len[b];
    DSA_CHECK(kv_raw >= 0 && kv_raw <= T_max);
    const int Tb = min(max(kv_raw, 0), T_max);
    r.start = n_sink;
    r.n_in = max(0, Tb - n_stream - n_sink);
    r.in = nullptr;
  } else {
    const int cnt_raw = in_cnt[b];
    DSA_CHECK(cnt_raw >= 0 && cnt_raw <= in_stride);
    r.start = 0;
    r.n_in = min(max(cnt_raw, 0), in_stride);
    r.in = in_idx + static_cast<size_t>(b) * in_stride;
  }
  return r;
}

// Chunks of at most this many tokens are scored from shared memory: the CTA copies all
// key rows of its chunks in one round (every KV head of a token is one contiguous run)
// and the tournaments read them there, instead of a chain of dependent row loads.  Such
// a CTA takes up to kMaxChunksPerCta chunks, so that a stage of many small chunks runs
// in about one wave.
constexpr int kSmemRowsMaxL = 4;
constexpr int kMaxChunksPerCta = 4;
constexpr int kRhoMax = 512;   // per-CTA head maxima: chunks per CTA x H_q

// shared-memory layout, the same on both sides: head maxima, positions, fp32 query
// rows (multi-row blocks), staged key rows
struct ScoreSmem {
  size_t pos, q, rows, total;
  __host__ __device__ ScoreSmem(bool rows_mode, bool explicit_list, int L, int C, bool qreg, int T_q,
                                int H_q, int D, size_t row_bytes) {
    pos = kRhoMax * sizeof(float);
    const size_t npos = rows_mode ? static_cast<size_t>(C) * L : (explicit_list ? L : 0);
    q = pos + ((npos + 3) & ~size_t(3)) * sizeof(int);
    size_t o = q + (qreg ? 0 : static_cast<size_t>(T_q) * H_q * D * sizeof(float));
    rows = (o + 15) & ~size_t(15);
    total = rows + (rows_mode ? static_cast<size_t>(C) * L * row_bytes : 0);
  }
};

// tournament levels whose candidate rows are requested from L2 ahead of time (a third
// level, four candidates of which a head probes one, measured slower)
constexpr int kWarmLevels = 2;

// NT_MAX / MIN_B: launch bounds.  Up to 32 query heads (256 threads) the kernel keeps
// eight CTAs (64 warps) resident per SM: every octet waits on one dependent key row at
// a time, so the number of tournaments in flight is what feeds HBM.
// TQ / TK: storage of the query (bf16 or fp32) and of the key rows (the same, or FP8
// E4M3 under a bf16 query).
// ROWS: the key rows of the CTA's C chunks (C * L <= kMaxChunksPerCta * kSmemRowsMaxL
// tokens) are staged in shared memory; otherwise C = 1 and the rows are read as the
// tournament needs them.
template <typename TQ, typename TK, int D, bool QREG, int NT_MAX, int MIN_B, bool ROWS>
__global__ void __launch_bounds__(NT_MAX, MIN_B) stage_score_kernel(StageScoreArgs a, int C) {
  constexpr int EPL = D / 8;
  if (!ROWS) C = 1;
  const size_t row_stride = static_cast<size_t>(a.H_kv) * D;   // elements per token
  extern __shared__ __align__(16) unsigned char smem[];
  float *s_rho = reinterpret_cast<float *>(smem);
  int *s_pos, *s_q_raw;
  uint4 *s_rows;
  {
    const ScoreSmem lay(ROWS, a.in_idx != nullptr, a.L, C, QREG, a.T_q, a.H_q, D, row_stride * sizeof(TK));
    s_pos = reinterpret_cast<int *>(smem + lay.pos);
    s_q_raw = reinterpret_cast<int *>(smem + lay.q);
    s_rows = reinterpret_cast<uint4 *>(smem + lay.rows);
  }
  float *s_q = reinterpret_cast<float *>(s_q_raw);

  grid_dep_wait();
  const int b = blockIdx.y, j0 = blockIdx.x * C;
  const TK *kbase = static_cast<const TK *>(a.k) + static_cast<size_t>(b) * a.T_max * row_stride;
  const int32_t *lst = a.in_idx ? a.in_idx + static_cast<size_t>(b) * a.in_stride : nullptr;
  // The list entries are read before the list's count, which only bounds what is used
  // below: a read stays inside the row of the list, and a position (possibly stale) is
  // clamped to the key rows.
  int pv = 0;
  if (ROWS) {
    // all heads of the C * L tokens, 16-byte asynchronous copies (all in flight at once)
    const int per_tok = static_cast<int>(row_stride * sizeof(TK) / 16);
    const int n_u = C * a.L * per_tok;
#pragma unroll 4
    for (int u = threadIdx.x; u < n_u; u += blockDim.x) {
      const int x = u / per_tok, w = u - x * per_tok;
      const int p = j0 * a.L + x;
      const int pos = lst ? min(max(__ldg(lst + min(p, a.in_stride - 1)), 0), a.T_max - 1)
                          : min(a.n_sink + p, a.T_max - 1);
      if (w == 0) s_pos[x] = pos;
      cp_async_16(s_rows + u, reinterpret_cast<const uint4 *>(kbase + static_cast<size_t>(pos) * row_stride) + w);
    }
    cp_async_commit();
  } else if (lst && static_cast<int>(threadIdx.x) < a.L) {
    pv = __ldg(lst + min(j0 * a.L + static_cast<int>(threadIdx.x), a.in_stride - 1));
  }
  const InputRange ir = stage_input(a.kv_len, b, a.T_max, a.n_sink, a.n_stream, a.in_idx,
                                    a.in_cnt, a.in_stride);
  const int n_chunk = (ir.n_in + a.L - 1) / a.L;
  if (j0 >= n_chunk) {
    if (ROWS) cp_async_wait<0>();   // no copy outlives the CTA
    return;
  }
  const TQ *q = static_cast<const TQ *>(a.q) + static_cast<size_t>(b) * a.T_q * a.H_q * D;
  if (!ROWS && ir.in) {
    const int len0 = min(a.L, ir.n_in - j0 * a.L);
    for (int x = threadIdx.x; x < len0; x += blockDim.x) {
      const int raw = x == static_cast<int>(threadIdx.x) ? pv : ir.in[j0 * a.L + x];
      DSA_CHECK(raw >= 0 && raw < a.T_max);   // a list entry (cached lists: as stored)
      s_pos[x] = min(max(raw, 0), a.T_max - 1);
    }
  }
  if (!QREG) {
    // the query rows as fp32, 16-byte loads, independent across the unrolled iterations
    // (a one-warp CTA loads T_q * H_q * D elements)
    const int n8 = a.T_q * a.H_q * D / 8;   // D is a multiple of 8
#pragma unroll 8
    for (int e = threadIdx.x; e < n8; e += blockDim.x) {
      float4 lo, hi;
      if constexpr (sizeof(TQ) == 2) {
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(q) + e);
        lo = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
        hi = make_float4(bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w));
      } else {
        lo = __ldg(reinterpret_cast<const float4 *>(q) + 2 * e);
        hi = __ldg(reinterpret_cast<const float4 *>(q) + 2 * e + 1);
      }
      reinterpret_cast<float4 *>(s_q)[2 * e] = lo;
      reinterpret_cast<float4 *>(s_q)[2 * e + 1] = hi;
    }
  }
  if (ROWS) cp_async_wait<0>();
  __syncthreads();

  // Octet o (eight lanes) scores for head o % H_q.  With several query rows and fewer
  // than four heads, the warp's spare octets take a share of the rows (octet o the rows
  // t = o / H_q (mod RS)) and the RS octets of a head combine their row maxima, so the
  // tournament of every head runs on all of them alike.
  const int oct = threadIdx.x >> 3, sub = threadIdx.x & 7;
  const int RS = QREG ? 1 : max(1, static_cast<int>(blockDim.x >> 3) / a.H_q);   // 4, 2 or 1 when T_q > 1
  const int h = QREG ? oct : oct % a.H_q, rs = QREG ? 0 : oct / a.H_q;
  const int G = a.H_q / a.H_kv;
  const int n_here = min(C, n_chunk - j0);   // chunks of this CTA that exist
  if (QREG ? h < a.H_q : rs < RS) {
    const int g = h / G;
    const unsigned omask = 0xffu << (threadIdx.x & 24);
    // the lanes of all RS octets of this head (RS > 1 only in one-warp CTAs)
    unsigned hmask = 0u;
    for (int r = 0; r < RS; ++r) hmask |= 0xffu << (8 * (h + r * a.H_q));
    if (RS == 1) hmask = omask;
    constexpr int NV = EPL * static_cast<int>(sizeof(TK)) / 16;    // 16-byte key loads per lane
    constexpr int NVQ = EPL * static_cast<int>(sizeof(TQ)) / 16;   // and query loads
    static_assert(NV >= 1, "a lane's key slice is at least 16 bytes");
    // the query slice stays in its storage format too (bf16 pairs or fp32)
    uint4 qraw[QREG ? NVQ : 1];
    if (QREG) {
      const uint4 *qp = reinterpret_cast<const uint4 *>(q + static_cast<size_t>(h) * D + sub * EPL);
#pragma unroll
      for (int i = 0; i < NVQ; ++i) qraw[i] = __ldg(qp + i);
    }
    const TK *kb = kbase + static_cast<size_t>(g) * D + sub * EPL;
    const int T_q = QREG ? 1 : a.T_q;
    for (int c = 0; c < n_here; ++c) {
      const int j = j0 + c;
      const int base = j * a.L;
      const int len = min(a.L, ir.n_in - base);
      // position of the chunk's x-th token
      auto pos_of = [&](int x) -> int {
        return ROWS ? s_pos[c * a.L + x] : (ir.in ? s_pos[x] : ir.start + base + x);
      };
      auto score = [&](int x) -> float {
        // keep the row as raw 16-byte words and widen while multiplying (fewer registers)
        uint4 raw[NV];
        if (ROWS) {
          const uint4 *kp = s_rows + (static_cast<size_t>(c * a.L + x) * row_stride +
                                      static_cast<size_t>(g) * D + sub * EPL) * sizeof(TK) / 16;
#pragma unroll
          for (int i = 0; i < NV; ++i) raw[i] = kp[i];
        } else {
          const uint4 *kp = reinterpret_cast<const uint4 *>(kb + static_cast<size_t>(pos_of(x)) * row_stride);
#pragma unroll
          for (int i = 0; i < NV; ++i) raw[i] = __ldg(kp + i);
        }
        float best = -INFINITY;
        for (int t = rs; t < T_q; t += RS) {
          const float *qq = s_q + (static_cast<size_t>(t) * a.H_q + h) * D + sub * EPL;
          float d = 0.f;
          if constexpr (std::is_same<TQ, TK>::value && sizeof(TK) == 2 && QREG) {
            // bf16 query and key words straight into a mixed-precision FMA (bf16 inputs
            // widened exactly, fp32 accumulate): the same products and order as widening
            // first, without the widening instructions
#pragma unroll
            for (int i = 0; i < NV; ++i) {
              d = fma_bf16x2_acc(qraw[i].x, raw[i].x, d);
              d = fma_bf16x2_acc(qraw[i].y, raw[i].y, d);
              d = fma_bf16x2_acc(qraw[i].z, raw[i].z, d);
              d = fma_bf16x2_acc(qraw[i].w, raw[i].w, d);
            }
          } else if constexpr (std::is_same<TQ, TK>::value) {
            constexpr int per = Store<TK>::kPer16;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
              float kf[per], qf[per];
              unpack16(raw[i], kf, TK());
              if (QREG) unpack16(qraw[i], qf, TQ());
#pragma unroll
              for (int e = 0; e < per; ++e) d = fmaf(QREG ? qf[e] : qq[i * per + e], kf[e], d);
            }
          } else {
            // FP8 keys under a bf16 query: each 32-bit key word is four elements, matched
            // by two 32-bit query words
#pragma unroll
            for (int i = 0; i < NV; ++i) {
              const uint32_t kw[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
              for (int wi = 0; wi < 4; ++wi) {
                const int e0 = 16 * i + 4 * wi;   // first element of this word in the slice
                // the word's four codes widened by the hardware conversion (E4M3 -> f16 ->
                // f32, both exact: the same values as a bit-level decode)
                float k4[4];
                f16x2_to_f32x2(e4m3x2_to_f16x2(kw[wi]), k4[0], k4[1]);
                f16x2_to_f32x2(e4m3x2_to_f16x2(kw[wi] >> 16), k4[2], k4[3]);
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) {
                  const float kf = k4[bb];
                  float qf;
                  if (QREG) {
                    const uint4 &qv = qraw[(e0 + bb) >> 3];
                    const int qw = ((e0 + bb) >> 1) & 3;
                    const uint32_t word = qw == 0 ? qv.x : qw == 1 ? qv.y : qw == 2 ? qv.z : qv.w;
                    qf = ((e0 + bb) & 1) ? bf16_hi(word) : bf16_lo(word);
                  } else {
                    qf = qq[e0 + bb];
                  }
                  d = fmaf(qf, kf, d);
                }
              }
            }
          }
          d += __shfl_xor_sync(omask, d, 4);
          d += __shfl_xor_sync(omask, d, 2);
          d += __shfl_xor_sync(omask, d, 1);
          best = fmaxf(best, d);
        }
        // the head's other octets hold the maxima of its other rows
        for (int o = 8 * a.H_q; o < 8 * a.H_q * RS; o <<= 1) best = fmaxf(best, __shfl_xor_sync(hmask, best, o));
        return best;
      };
      // The first kWarmLevels probes of every head's tournament can only be one of the
      // 2^level - 1 midpoints of the first levels (the same for every head of the
      // chunk): ask L2 for those rows now, in the round of the first load, so those
      // levels' loads hit L2 instead of each waiting a DRAM round.
      auto warm = [&]() {
        constexpr int kNodes = (1 << kWarmLevels) - 1;
        int los[kNodes], his[kNodes];   // candidate ranges, heap order (children 2i+1, 2i+2)
        los[0] = 0;
        his[0] = len - 1;
#pragma unroll
        for (int i = 0; i < kNodes; ++i) {
          if (los[i] < his[i]) {
            const int mid = (los[i] + his[i] + 1) >> 1;
            const char *row = reinterpret_cast<const char *>(kb + static_cast<size_t>(pos_of(mid)) * row_stride);
            asm volatile("prefetch.global.L2 [%0];\n" ::"l"(row));
            if (2 * i + 2 < kNodes) {
              los[2 * i + 1] = los[i];
              his[2 * i + 1] = mid - 1;
              los[2 * i + 2] = mid;
              his[2 * i + 2] = his[i];
            }
          } else if (2 * i + 2 < kNodes) {
            los[2 * i + 1] = los[2 * i + 2] = 1;   // empty
            his[2 * i + 1] = his[2 * i + 2] = 0;
          }
        }
      };
      if constexpr (kWarmLevels > 0 && !ROWS) {
        if ((sub & 3) == 0 && rs == 0) warm();   // two lanes per row: one per 128-byte line
      }
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
      if (sub == 0 && rs == 0) {
        s_rho[c * a.H_q + h] = s_lo;
        if (a.dbg_rep) {
          const size_t o = (static_cast<size_t>(b) * a.H_q + h) * a.max_chunks + j;
          a.dbg_rep[o] = pos_of(lo);
          if (a.dbg_rho) a.dbg_rho[o] = s_lo;
        }
      }
    }
  }
  __syncthreads();
  // chunk score: max over all query heads (and rows, already inside s_rho), one warp
  // per chunk
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int c = warp; c < n_here; c += blockDim.x >> 5) {
    float m = -INFINITY;
    for (int i = lane; i < a.H_q; i += 32) m = fmaxf(m, s_rho[c * a.H_q + i]);
    m = warp_max(m);
    if (lane == 0) a.score[static_cast<size_t>(b) * a.max_chunks + j0 + c] = m;
  }
}

constexpr int kTopkThreads = 1024;

__global__ void __launch_bounds__(kTopkThreads) stage_topk_kernel(StageTopkArgs a) {
  constexpr int NT = kTopkThreads;
  extern __shared__ int s_chunk_of_rank[];   // [K]
  __shared__ uint32_t s_hist[256];
  __shared__ uint32_t s_res[2];
  __shared__ int s_warp[NT / 32 + 1];
  if (a.release_dependents) grid_dep_release();
  grid_dep_wait();
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

// Register-resident top-K for up to kFastNT * kFastNPT chunks.  Thread t owns the
// kFastNPT consecutive chunks starting at t * kFastNPT, so one block-wide scan of
// per-thread counts ranks the kept chunks in index order.
// Selection: the ordered keys are spread over kFastNB buckets by a map that never
// decreases with the key (equal keys share a bucket; a higher bucket holds only
// larger keys).  One histogram and one scan find the bucket holding the K-th largest
// key; only that bucket's members (usually a handful) are ranked exactly, by key and
// then by chunk index.  When more than kFastCand keys share the boundary bucket (many
// equal scores), an 8-bit radix select over the resident keys decides instead.
constexpr int kFastNT = 1024;
constexpr int kFastNPT = 16;
constexpr int kFastNB = 4096;
constexpr int kFastCand = 1024;
constexpr int kTopkMaxParts = 8;         // CTAs writing one row's list
constexpr int kTopkPartEntries = 2048;   // list entries per part, at least

// inclusive block scan of one value per thread (thread order); all threads call it.
// One barrier: every warp reads all warp totals and forms its own offset.  Two scans in
// a row must use different s_w buffers (a slow warp may still read the first).
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t v, uint32_t *s_w, uint32_t *total) {
  static_assert(kFastNT == 1024, "one warp total per lane");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) s_w[warp] = incl;
  __syncthreads();
  const uint32_t x = s_w[lane];
  *total = __reduce_add_sync(kFull, x);
  return __reduce_add_sync(kFull, lane < warp ? x : 0u) + incl;
}

// POW2: 16-byte access to the score row and the token lists (see the host side).
// NPT: chunks per thread, the smallest power of two with kFastNT * NPT >= max_chunks,
// so that no thread walks empty slots.
template <bool POW2, int NPT>
__global__ void __launch_bounds__(kFastNT) stage_topk_fast_kernel(StageTopkArgs a) {
  constexpr int NT = kFastNT, NB = kFastNB;
  extern __shared__ int s_chunk_of_rank[];   // [K]
  __shared__ uint32_t s_hist[NB];
  __shared__ uint32_t s_ckey[kFastCand];
  __shared__ int s_cidx[kFastCand];
  __shared__ uint32_t s_keep[(NT * NPT + 31) / 32];   // kept bits of boundary-bucket chunks
  __shared__ uint32_t s_w[3][NT / 32];   // one buffer per block scan
  __shared__ uint32_t s_misc[8];   // 0 min, 1 max, 2 boundary bucket, 3 count above, 4 candidates
  __shared__ uint32_t s_hist8[256];
  __shared__ uint32_t s_res[2];
  if (a.release_dependents) grid_dep_release();
  grid_dep_wait();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i0 = tid * NPT;
  // the row's scores come in while the candidate range is read (slots past the row's
  // chunk count are ignored below)
  const float *sc = a.score + static_cast<size_t>(b) * a.max_chunks;
  float sv[NPT];
  if (POW2 && NPT % 4 == 0 && i0 + NPT <= a.max_chunks) {
#pragma unroll
    for (int k = 0; k < NPT; k += 4) {
      const float4 f = __ldg(reinterpret_cast<const float4 *>(sc + i0 + k));
      sv[k] = f.x;
      sv[k + 1] = f.y;
      sv[k + 2] = f.z;
      sv[k + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < NPT; ++k) sv[k] = i0 + k < a.max_chunks ? __ldg(sc + i0 + k) : 0.f;
  }
  const InputRange ir = stage_input(a.kv_len, b, a.T_max, a.n_sink, a.n_stream, a.in_idx,
                                    a.in_cnt, a.in_stride);
  const int L = a.L;
  const int n_chunk = min((ir.n_in + L - 1) / L, a.max_chunks);
  const bool keep_all = n_chunk <= a.K;
  uint32_t key[NPT];
#pragma unroll
  for (int k = 0; k < NPT; ++k) key[k] = (i0 + k < n_chunk) ? ordered_key(sv[k]) : 0u;
  uint32_t kept_bits = 0u;   // bit k: chunk i0 + k is kept
  if (keep_all) {
#pragma unroll
    for (int k = 0; k < NPT; ++k)
      if (i0 + k < n_chunk) kept_bits |= 1u << k;
  } else {
    // key range of the row
    uint32_t mn = 0xffffffffu, mx = 0u;
#pragma unroll
    for (int k = 0; k < NPT; ++k) {
      if (i0 + k < n_chunk) {
        mn = min(mn, key[k]);
        mx = max(mx, key[k]);
      }
    }
    mn = __reduce_min_sync(kFull, mn);
    mx = __reduce_max_sync(kFull, mx);
    for (int i = tid; i < NB; i += NT) s_hist[i] = 0u;
    for (int i = tid; i < (NT * NPT + 31) / 32; i += NT) s_keep[i] = 0u;
    if (lane == 0) {
      s_hist8[warp] = mn;          // scratch for the block reduction
      s_hist8[32 + warp] = mx;
    }
    if (tid == 0) s_misc[4] = 0u;
    __syncthreads();
    // every warp reduces the 32 warp partials itself (no second barrier)
    const uint32_t kmin = __reduce_min_sync(kFull, s_hist8[lane]);
    const uint32_t kmax = __reduce_max_sync(kFull, s_hist8[32 + lane]);
    const float bscale = static_cast<float>(NB) / (static_cast<float>(kmax - kmin) + 1.0f);
    // never decreasing in the key: a uint32 -> float conversion keeps order (ties at
    // worst), as do the positive scaling and the truncation
    auto bucket = [&](uint32_t u) {
      return min(NB - 1, static_cast<int>(static_cast<float>(u - kmin) * bscale));
    };
#pragma unroll
    for (int k = 0; k < NPT; ++k)
      if (i0 + k < n_chunk) atomicAdd(&s_hist[bucket(key[k])], 1u);
    __syncthreads();
    // thread t holds buckets NB-1-4t .. NB-4-4t; counts from the top bucket down
    uint32_t c4[4], sum4 = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      c4[j] = s_hist[NB - 1 - 4 * tid - j];
      sum4 += c4[j];
    }
    uint32_t total;
    const uint32_t incl = block_incl_scan(sum4, s_w[0], &total);
    const uint32_t K = static_cast<uint32_t>(a.K);
    if (incl - sum4 < K && K <= incl) {
      uint32_t run = incl - sum4;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (run + c4[j] >= K) {
          s_misc[2] = static_cast<uint32_t>(NB - 1 - 4 * tid - j);
          s_misc[3] = run;
          s_misc[5] = c4[j];
          break;
        }
        run += c4[j];
      }
    }
    __syncthreads();
    const int bstar = static_cast<int>(s_misc[2]);
    const uint32_t above = s_misc[3];
    if (s_misc[5] == K - above) {
      // the whole boundary bucket is in the top K (the usual case: one key there)
#pragma unroll
      for (int k = 0; k < NPT; ++k)
        if (i0 + k < n_chunk && bucket(key[k]) >= bstar) kept_bits |= 1u << k;
    } else {
      // the boundary bucket's members
#pragma unroll
      for (int k = 0; k < NPT; ++k) {
        const bool valid = i0 + k < n_chunk;
        const int bk = valid ? bucket(key[k]) : -1;
        if (bk > bstar) kept_bits |= 1u << k;
        // one slot claim per warp and key position
        const unsigned members = __ballot_sync(kFull, bk == bstar);
        if (members) {
          uint32_t base = 0;
          if (lane == __ffs(members) - 1) base = atomicAdd(&s_misc[4], static_cast<uint32_t>(__popc(members)));
          base = __shfl_sync(kFull, base, __ffs(members) - 1);
          if (bk == bstar) {
            const uint32_t slot = base + __popc(members & ((1u << lane) - 1u));
            if (slot < static_cast<uint32_t>(kFastCand)) {
              s_ckey[slot] = key[k];
              s_cidx[slot] = i0 + k;
            }
          }
        }
      }
      __syncthreads();
      const uint32_t m = s_misc[4];
      if (m <= static_cast<uint32_t>(kFastCand)) {
        // exact ranks inside the bucket: larger key first, then smaller chunk index
        const uint32_t need = K - above;   // 1 <= need <= m
        for (uint32_t j = tid; j < m; j += NT) {
          const uint32_t kj = s_ckey[j];
          const int ij = s_cidx[j];
          uint32_t rank = 0;
          for (uint32_t i = 0; i < m; ++i) {
            const uint32_t ki = s_ckey[i];
            rank += (ki > kj || (ki == kj && s_cidx[i] < ij)) ? 1u : 0u;
          }
          if (rank < need) atomicOr(&s_keep[ij >> 5], 1u << (ij & 31));
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < NPT; ++k) {
          const int i = i0 + k;
          if (i < n_chunk && bucket(key[k]) == bstar && ((s_keep[i >> 5] >> (i & 31)) & 1u))
            kept_bits |= 1u << k;
        }
      } else {
        // many equal or nearly equal keys: radix select over the resident keys for the
        // K-th largest key `thr` and the number `k_eq` of its copies in the top K, then
        // keep the first k_eq copies in index order
        uint32_t prefix = 0u, mask = 0u, k_rem = K;
        for (int pass = 0; pass < 4; ++pass) {
          const int shift = 24 - 8 * pass;
          for (int i = tid; i < 256; i += NT) s_hist8[i] = 0u;
          __syncthreads();
#pragma unroll
          for (int k = 0; k < NPT; ++k) {
            const bool ok = i0 + k < n_chunk && (key[k] & mask) == prefix;
            const uint32_t bin = ok ? ((key[k] >> shift) & 255u) : 256u;
            const unsigned peers = __match_any_sync(kFull, bin);
            if (ok && lane == __ffs(peers) - 1) atomicAdd(&s_hist8[bin], static_cast<uint32_t>(__popc(peers)));
          }
          __syncthreads();
          if (warp == 0) {
            const int top = 255 - lane * 8;
            uint32_t c[8], sum = 0;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              c[t] = s_hist8[top - t];
              sum += c[t];
            }
            uint32_t inc = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const uint32_t v = __shfl_up_sync(kFull, inc, o);
              if (lane >= o) inc += v;
            }
            const uint32_t exc = inc - sum;
            if (exc < k_rem && k_rem <= inc) {
              uint32_t run = exc;
#pragma unroll
              for (int t = 0; t < 8; ++t) {
                if (run + c[t] >= k_rem) {
                  s_res[0] = static_cast<uint32_t>(top - t);
                  s_res[1] = run;
                  break;
                }
                run += c[t];
              }
            }
          }
          __syncthreads();
          prefix |= s_res[0] << shift;
          mask |= 255u << shift;
          k_rem -= s_res[1];
          __syncthreads();
        }
        const uint32_t thr = prefix, k_eq = k_rem;
        uint32_t eq = 0;
#pragma unroll
        for (int k = 0; k < NPT; ++k) eq += (i0 + k < n_chunk && key[k] == thr) ? 1u : 0u;
        uint32_t tot_eq;
        uint32_t eq_b = block_incl_scan(eq, s_w[1], &tot_eq) - eq;
        kept_bits = 0u;
#pragma unroll
        for (int k = 0; k < NPT; ++k) {
          if (i0 + k < n_chunk) {
            if (key[k] > thr) kept_bits |= 1u << k;
            if (key[k] == thr) {
              if (eq_b < k_eq) kept_bits |= 1u << k;
              ++eq_b;
            }
          }
        }
      }
    }
  }
  // ranks of the kept chunks in index order
  const uint32_t nk = static_cast<uint32_t>(__popc(kept_bits));
  uint32_t tot_kept;
  uint32_t r = block_incl_scan(nk, s_w[2], &tot_kept) - nk;
#pragma unroll
  for (int k = 0; k < NPT; ++k) {
    if ((kept_bits >> k) & 1u) {
      if (r < static_cast<uint32_t>(a.K)) s_chunk_of_rank[r] = i0 + k;
      ++r;
    }
  }
  __syncthreads();
  const int n_kept = min(static_cast<int>(tot_kept), max(a.K, 0));
  int count = n_kept * L;
  // only the last chunk of the list can be short; kept, it has the highest rank
  if (n_kept > 0 && s_chunk_of_rank[n_kept - 1] == n_chunk - 1) count -= n_chunk * L - ir.n_in;
  int32_t *out = a.out_idx + static_cast<size_t>(b) * a.out_stride;
  int32_t *dbg = a.dbg_idx ? a.dbg_idx + static_cast<size_t>(b) * a.out_stride : nullptr;
  // this CTA's part of the list (every part repeats the selection above)
  const int part_len = (((a.out_stride + gridDim.y - 1) / gridDim.y) + 3) & ~3;
  const int e_beg = min(a.out_stride, static_cast<int>(blockIdx.y) * part_len);
  const int e_end = min(a.out_stride, e_beg + part_len);
  if (POW2 && (L & 3) == 0 && (a.out_stride & 3) == 0) {
    // four consecutive entries share a chunk: 16-byte loads and stores, kU gathers in
    // flight per thread before their stores
    constexpr int kU = 4;
    const int lg = __ffs(L) - 1;
    for (int e0 = e_beg + 4 * tid; e0 < e_end; e0 += 4 * NT * kU) {
      int4 val[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int e = e0 + 4 * NT * u;
        val[u] = make_int4(-1, -1, -1, -1);
        if (e < count) {
          const int rr = e >> lg, x = e & (L - 1);
          const int src = (s_chunk_of_rank[rr] << lg) + x;
          if (ir.in) {
            val[u] = *reinterpret_cast<const int4 *>(ir.in + src);
          } else {
            val[u] = make_int4(ir.start + src, ir.start + src + 1, ir.start + src + 2, ir.start + src + 3);
          }
          if (e + 1 >= count) val[u].y = -1;
          if (e + 2 >= count) val[u].z = -1;
          if (e + 3 >= count) val[u].w = -1;
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int e = e0 + 4 * NT * u;
        if (e < e_end) {
          *reinterpret_cast<int4 *>(out + e) = val[u];
          if (dbg) *reinterpret_cast<int4 *>(dbg + e) = val[u];
        }
      }
    }
  } else {
    for (int e = e_beg + tid; e < e_end; e += NT) {
      int val = -1;
      if (e < count) {
        const int rr = e / L, x = e - rr * L;
        const int src = s_chunk_of_rank[rr] * L + x;
        val = ir.in ? ir.in[src] : ir.start + src;
      }
      out[e] = val;
      if (dbg) dbg[e] = val;
    }
  }
  if (tid == 0 && blockIdx.y == 0) {
    a.out_cnt[b] = count;
    if (a.dbg_cnt) a.dbg_cnt[b] = count;
  }
}

template <typename TQ, typename TK, int D>
cudaError_t launch_score_t(const StageScoreArgs &a, cudaStream_t s) {
  const bool explicit_list = a.in_idx != nullptr;
  const bool qreg = a.T_q == 1;
  const int threads = ((8 * a.H_q + 31) / 32) * 32;
  if (a.max_chunks == 0) return cudaSuccess;
  // fp32 rows need twice the registers: six CTAs per SM there; the staged-rows variant
  // loops over its chunks and keeps two CTAs fewer
  constexpr int kMinB = sizeof(TQ) == 2 ? 8 : 6;
  constexpr int kMinBRows = kMinB - 2;
  const size_t row_bytes = static_cast<size_t>(a.H_kv) * D * sizeof(TK);
  constexpr size_t kRowsSmemMax = 64 * 1024;   // staged rows per CTA
  constexpr size_t kSmemPerSm = 228 * 1024;     // 1 KB of it reserved per CTA
  const bool rows = a.L <= kSmemRowsMaxL && (!qreg || threads <= 256) && a.L * row_bytes <= kRowsSmemMax;
  int C = 1;
  if (rows) {
    // The fewest chunks per CTA that hold the whole stage in one wave of resident CTAs
    // (registers and shared memory both bound the CTAs per SM); failing that, the most
    // chunks in flight.
    int dev = 0, n_sm = 0;   // the current device's (a process may drive several)
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    n_sm = std::max(n_sm, 1);
    const long long need = static_cast<long long>(a.B) * a.max_chunks;
    long long best = -1;
    for (int c = 1; c <= kMaxChunksPerCta; ++c) {
      if (c * a.H_q > kRhoMax || c * a.L * row_bytes > kRowsSmemMax) break;
      const size_t bytes = ScoreSmem(true, explicit_list, a.L, c, qreg, a.T_q, a.H_q, D, row_bytes).total;
      const long long per_sm = std::min<long long>(qreg ? kMinBRows : 1, (kSmemPerSm / (bytes + 1024)));
      const long long cap = static_cast<long long>(n_sm) * per_sm * c;
      if (cap > best) {
        best = cap;
        C = c;
      }
      if (cap >= need) break;
    }
  }
  const ScoreSmem lay(rows, explicit_list, a.L, C, qreg, a.T_q, a.H_q, D, row_bytes);
  const size_t smem = lay.total;
  dim3 grid((a.max_chunks + C - 1) / C, a.B);
  auto go = [&](auto kern) {
    if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch_pdl(kern, grid, dim3(threads), smem, s, a, C);
  };
  if (qreg && threads <= 256) {
    if (rows) go(stage_score_kernel<TQ, TK, D, true, 256, kMinBRows, true>);
    else go(stage_score_kernel<TQ, TK, D, true, 256, kMinB, false>);
  } else if (qreg) {
    go(stage_score_kernel<TQ, TK, D, true, 1024, 1, false>);
  } else {
    if (rows) go(stage_score_kernel<TQ, TK, D, false, 1024, 1, true>);
    else go(stage_score_kernel<TQ, TK, D, false, 1024, 1, false>);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_stage_score(const StageScoreArgs &a, cudaStream_t s) {
  if (stage_score_tc_ok(a)) return launch_stage_score_tc(a, s);
  if (a.dtype == DSA_BF16_FP8KV) return launch_score_t<uint16_t, Fp8E4M3, 128>(a, s);   // D = 128
  if (a.dtype == DSA_BF16) {
    return a.D == 128 ? launch_score_t<uint16_t, uint16_t, 128>(a, s)
                      : launch_score_t<uint16_t, uint16_t, 64>(a, s);
  }
  return a.D == 128 ? launch_score_t<float, float, 128>(a, s) : launch_score_t<float, float, 64>(a, s);
}

cudaError_t launch_stage_topk(const StageTopkArgs &a, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(a.K) * sizeof(int);
  // static shared memory: about 28 KB in the register-resident kernel, 1 KB otherwise
  // The register-resident kernel spreads the list writes over `parts` CTAs per row,
  // each repeating the (cheap, deterministic) selection: one SM alone writes a list of
  // tens of thousands of entries at a fraction of the L2 bandwidth.
  const int parts = std::max(1, std::min(kTopkMaxParts, (a.out_stride + kTopkPartEntries - 1) / kTopkPartEntries));
  auto go = [&](auto kern, int threads, size_t static_bytes, int nparts) {
    if (smem + static_bytes > 48 * 1024)
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch_pdl(kern, dim3(a.B, nparts), dim3(threads), smem, s, a);
  };
  // 16-byte list access needs 16-byte aligned rows of the explicit input list, and rows
  // holding whole chunks (the last chunk's 16-byte groups then stay inside the row)
  const bool pow2 = (a.L & (a.L - 1)) == 0 && (reinterpret_cast<uintptr_t>(a.score) & 15) == 0 &&
                    (a.max_chunks & 3) == 0 &&
                    (a.in_idx == nullptr ||
                     ((reinterpret_cast<uintptr_t>(a.in_idx) & 15) == 0 && (a.in_stride & 3) == 0 &&
                      a.in_stride % a.L == 0)) &&
                    (reinterpret_cast<uintptr_t>(a.out_idx) & 15) == 0 &&
                    (a.dbg_idx == nullptr || (reinterpret_cast<uintptr_t>(a.dbg_idx) & 15) == 0);
  if (a.max_chunks <= kFastNT * kFastNPT) {
    auto pick = [&](auto pw) {
      constexpr bool P = decltype(pw)::value;
      if (a.max_chunks <= kFastNT) go(stage_topk_fast_kernel<P, 1>, kFastNT, 28 * 1024, parts);
      else if (a.max_chunks <= 2 * kFastNT) go(stage_topk_fast_kernel<P, 2>, kFastNT, 28 * 1024, parts);
      else if (a.max_chunks <= 4 * kFastNT) go(stage_topk_fast_kernel<P, 4>, kFastNT, 28 * 1024, parts);
      else if (a.max_chunks <= 8 * kFastNT) go(stage_topk_fast_kernel<P, 8>, kFastNT, 28 * 1024, parts);
      else go(stage_topk_fast_kernel<P, 16>, kFastNT, 28 * 1024, parts);
    };
    if (pow2) pick(std::true_type{});
    else pick(std::false_type{});
  } else {
    go(stage_topk_kernel, kTopkThreads, 2 * 1024, 1);
  }
  return cudaGetLastError();
}

}  // namespace dsa
