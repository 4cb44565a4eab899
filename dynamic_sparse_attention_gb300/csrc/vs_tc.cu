// MInference vertical-slash estimate on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// Source: "MInference 1.0: Accelerating Pre-filling for Long-Context LLMs via Dynamic
// Sparse Attention" (paper-graph-ui summary), section 3.4 "Online Dynamic Index
// Estimation: Vertical-Slash Heads" (Alg. 2 steps 1-3): the softmax of the last
// r = min(last_q, S) queries against every key (causal), its column sums (vertical)
// and its sums along the diagonals o = query position - key position (slash).
//
// Each CTA serves one KV head g of one batch row and a contiguous run of key tiles;
// its A/B operands are the G query heads of g (the 64 positions S-64 .. S-1 per head,
// loaded once by TMA; rows before the estimate window and keys after a row's position
// are masked) and the run's key tiles (TMA ring).  One thread issues the MMAs into
// double-buffered TMEM accumulators, epilogue warps read them.
//
//  pass 0 (row statistics): S = Q K^T with the query rows on the TMEM lanes (M = 128:
//    two heads of 64 rows per MMA), keys along the columns.  One thread per row keeps an
//    online maximum and sum of exp2 over its keys; the run's partial (max, sum) per row
//    goes to the workspace and a small kernel combines the runs.
//  pass 1 (sums): S^T = K Q^T with the keys on the TMEM lanes (M = 128 keys) and all
//    G x 64 query rows along the columns, so one thread owns one key: its column sum
//    over a head's 64 rows is a sum inside the thread, and each probability goes to
//    the diagonal u = row - key + 127 of the tile with a shared-memory reduction: the 32
//    lanes of a warp hit 32 different diagonals (no conflicts), and every warp adds
//    into its own accumulator in program order, so the per-tile diagonal partials come
//    out the same on every run.  A combine kernel adds the (at most two) tiles of every
//    offset in ascending tile order.
// Probabilities are exp2(s * scale * log2 e - c) with c = max + log2(sum) of the row
// (the base-2 logits of pass 0), i.e. the normalised softmax.  Every mbarrier wait is
// bounded: a CTA that gives up stops, drains its copies and MMAs, frees TMEM and sets
// an error word that dsa_device_error reports.
#include <math.h>

#include <atomic>
#include <cstring>

#include "api_common.h"
#include "common.cuh"
#include "launch.h"
#include "profile.h"
#include "tc_ptx.cuh"

namespace dsa {

static __device__ int g_vs_tc_error;   // sticky error word, read by dsa_device_error
// wait limit of the bounded waits (dsa_set_wait_limit; default half a second)
static __device__ unsigned long long g_vs_wait_limit_ns = 500000000ull;

namespace {

using namespace tc;

constexpr int kBoxRows = 64;          // query positions per head (S - 64 .. S - 1)
constexpr int kTile1 = 128;           // keys per tile in pass 1 (TMEM lanes)
constexpr int kDiag1 = kTile1 + kBoxRows - 1;   // diagonals one pass-1 tile touches
constexpr int kMaxStages = 3;         // key-tile ring (two where shared memory is short)
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

struct VsTcArgs {
  CUtensorMap tq, tk;
  int B, S, H_q, H_kv, G, D, r_q;
  int kt;                 // keys per tile of this pass
  int n_ktile, tiles_per_split, n_split;
  float sl2;
  float *part_m, *part_l;           // pass 0 out: [B, H_kv, n_split * khalves, G * 64]
  const float *row_m, *row_l;       // pass 1 in: [B, H_q, 64] (base-2 logits)
  float *vsum;                      // pass 1 out: [B, H_q, S]
  float *slash_part;                // pass 1 out: [B, H_q, n_ktile, kDiag1, 2 row halves]
};

// shared-memory layout (1024-byte aligned base).  Pass 1 also holds the probabilities
// of `nph` heads of one tile ([head][64 rows][128 keys] fp32) for the diagonal sums;
// the key ring and nph shrink, in that order, until everything fits.
struct TcLayout {
  uint32_t halves, q_half, k_half, k_stage, stages, nph;
  uint32_t oQ, oK, oBar, oMisc, oC, oP, oV, total;
  __host__ __device__ TcLayout(int G, int D, int kt, int pass) {
    halves = D / 64;
    const int slots = pass == 0 ? ((G + 1) / 2) * 2 : G;   // pass 0 pads to pairs of heads
    q_half = static_cast<uint32_t>(slots) * kBoxRows * 128;
    k_half = static_cast<uint32_t>(kt) * 128;
    k_stage = halves * k_half;
    const uint32_t p_head = kBoxRows * kTile1 * 4;
    const uint32_t fixed = halves * q_half + 64 * 8 + 64 + static_cast<uint32_t>(G) * kBoxRows * 4 + 4 * kTile1 * 4 + 1024;
    const uint32_t budget = 227u * 1024u;
    stages = kMaxStages;
    nph = pass == 1 ? (G >= 2 ? 2u : 1u) : 0u;
    while (fixed + stages * k_stage + nph * p_head > budget) {
      if (stages > 2) --stages;
      else if (nph > 1) --nph;
      else if (stages > 1) --stages;
      else break;
    }
    oQ = 0;
    oK = oQ + halves * q_half;
    oBar = oK + stages * k_stage;
    oMisc = oBar + 64 * 8;
    oC = oMisc + 64;                                        // pass 1: c per (head, row)
    oP = oC + static_cast<uint32_t>(G) * kBoxRows * 4;      // pass 1: probabilities
    oV = oP + nph * p_head;                                 // pass 1: [2 heads][2 row halves][128] column sums
    total = oV + (pass == 1 ? 4u * kTile1 * 4u : 0u);
  }
};

struct Waiter {
  volatile int *abort;
  __device__ bool operator()(uint64_t *bar, uint32_t parity) const {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    const uint64_t limit = g_vs_wait_limit_ns;
    const uint32_t hint = limit < 20000ull ? static_cast<uint32_t>(limit) : 20000u;
    while (true) {
      if (mbar_try_wait_hint(bar, parity, hint)) return true;
      if (*abort) return false;
      if (global_ns() - t0 > limit) {
        *abort = 1;
        return false;
      }
    }
  }
};

__device__ __forceinline__ bool drain(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > 200000000ull) return false;
  return true;
}

// warp-uniform bounded wait (lane 0 waits, the warp learns the outcome)
__device__ __forceinline__ bool warp_wait(const Waiter &w, uint64_t *bar, uint32_t parity) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = w(bar, parity) ? 1 : 0;
  ok = __shfl_sync(kFull, ok, 0);
  return ok != 0;
}

// 2^x with the hardware approximation (relative error about 2^-22; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

template <int PASS>
__global__ void __launch_bounds__(640, 1) vs_tc_kernel(const __grid_constant__ VsTcArgs a) {
  const TcLayout L(a.G, a.D, a.kt, PASS);
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.oBar);
  const int kStages = static_cast<int>(L.stages);
  uint64_t *k_full = bars, *k_empty = bars + kMaxStages;
  uint64_t *s_full = bars + 2 * kMaxStages, *s_empty = s_full + 2;
  uint64_t *q_full = s_empty + 2, *fin = q_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L.oMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L.oMisc + 4);
  // set only by epilogue warps, before the barrier that follows their wait for a tile
  volatile int *epi_abort = reinterpret_cast<volatile int *>(sm + L.oMisc + 8);
  const Waiter wt{abort_flag};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_epi = (blockDim.x >> 5) - 4;   // epilogue warps: 4 .. 4 + n_epi - 1
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int G = a.G, S = a.S;
  const int t_begin = split * a.tiles_per_split;
  const int t_end = min(a.n_ktile, t_begin + a.tiles_per_split);
  const int n_t = max(0, t_end - t_begin);
  // TMEM buffers: pass 0 always two of 256 columns; pass 1 two of G*64 columns when
  // they fit, else one of 512
  const int n_buf = PASS == 0 ? 2 : (G <= 4 ? 2 : 1);
  const uint32_t buf_cols = PASS == 0 ? 256u : (G <= 4 ? 256u : 512u);

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], n_epi);
    }
    mbar_init(q_full, 1);
    mbar_init(fin, 1);
    *abort_flag = 0;
    *epi_abort = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (PASS == 1) {
    // c = max + log2(sum) per (head slot, box row); rows outside the estimate: +inf
    float *cst = reinterpret_cast<float *>(sm + L.oC);
    for (int e = tid; e < G * kBoxRows; e += blockDim.x) {
      const int hs = e / kBoxRows, br = e - hs * kBoxRows;
      const int i = br - (kBoxRows - a.r_q);   // estimate row
      float c = INFINITY;
      if (i >= 0) {
        const size_t o = (static_cast<size_t>(b) * a.H_q + g * G + hs) * kBoxRows + i;
        const float m = a.row_m[o], l = a.row_l[o];
        if (m != -INFINITY && l > 0.f) c = m + log2f(l);
      }
      cst[e] = c;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    int issued = 0;
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, L.halves * static_cast<uint32_t>(G) * kBoxRows * 128);
      for (int hs = 0; hs < G; ++hs)
        for (uint32_t hh = 0; hh < L.halves; ++hh)
          tma_load_4d(sm + L.oQ + hh * L.q_half + hs * kBoxRows * 128, &a.tq, q_full, 64 * hh,
                      g * G + hs, S - kBoxRows, b);
      for (int i = 0; i < n_t; ++i) {
        const int st = i % kStages;
        if (i >= kStages && !wt(&k_empty[st], ((i / kStages) - 1) & 1)) break;
        mbar_arrive_expect_tx(&k_full[st], L.k_stage);
        for (uint32_t hh = 0; hh < L.halves; ++hh)
          tma_load_4d(sm + L.oK + st * L.k_stage + hh * L.k_half, &a.tk, &k_full[st], 64 * hh, g,
                      (t_begin + i) * a.kt, b);
        ++issued;
      }
      if (*abort_flag) {
        // let this CTA's bulk copies land before it exits
        for (int i = max(0, issued - kStages); i < issued; ++i) drain(&k_full[i % kStages], (i / kStages) & 1);
        drain(q_full, 0);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t sQ = smem_u32(sm + L.oQ), sK = smem_u32(sm + L.oK);
      bool ok = wt(q_full, 0);
      for (int i = 0; ok && i < n_t; ++i) {
        const int st = i % kStages, buf = i % n_buf;
        if (!(ok = wt(&k_full[st], (i / kStages) & 1))) break;
        if (i >= n_buf && !(ok = wt(&s_empty[buf], ((i / n_buf) - 1) & 1))) break;
        tc_fence_after();
        const uint32_t d0 = tmem + static_cast<uint32_t>(buf) * buf_cols;
        const uint32_t kst = sK + st * L.k_stage;
        if (PASS == 0) {
          // D[slot s] (128 rows x kt keys) = Q rows of heads 2s, 2s+1 x K^T
          const uint32_t id = idesc_bf16_f32(128, a.kt, false, false);
          const int n_slot = (G + 1) / 2;
          for (int s = 0; s < n_slot; ++s)
            for (int kk = 0; kk < a.D / 16; ++kk) {
              const uint64_t ad = sdesc_sw128(sQ + (kk >> 2) * L.q_half + s * 2 * kBoxRows * 128 + (kk & 3) * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(kst + (kk >> 2) * L.k_half + (kk & 3) * 32, 16, 1024);
              tc_mma(d0 + static_cast<uint32_t>(s * a.kt), ad, bd, id, kk > 0 ? 1u : 0u);
            }
        } else {
          // D (128 keys x up to 256 query rows per MMA) = K x Q^T
          for (int part = 0; part * 4 < G; ++part) {
            const int rows = 64 * min(4, G - 4 * part);
            const uint32_t id = idesc_bf16_f32(128, rows, false, false);
            for (int kk = 0; kk < a.D / 16; ++kk) {
              const uint64_t ad = sdesc_sw128(kst + (kk >> 2) * L.k_half + (kk & 3) * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(sQ + (kk >> 2) * L.q_half + part * 4 * kBoxRows * 128 + (kk & 3) * 32, 16, 1024);
              tc_mma(d0 + static_cast<uint32_t>(part * 256), ad, bd, id, kk > 0 ? 1u : 0u);
            }
          }
        }
        tc_commit(&s_full[buf]);
        tc_commit(&k_empty[st]);
      }
      tc_commit(fin);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    const int e = warp - 4;
    const int quarter = warp & 3;   // TMEM lanes this warp may access
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    if (PASS == 0) {
      // warp e: head pair slot (e >> 2) % n_slot, key half e / (4 n_slot) of every tile
      const int n_slot = (G + 1) / 2;
      const int slot = (e >> 2) % n_slot;
      const int kh = e / (4 * n_slot), nkh = n_epi / (4 * n_slot);
      const int kw = a.kt / nkh;                    // keys of a tile this warp reads
      const int row = quarter * 32 + lane;          // row of the pair
      const int hs = 2 * slot + (row >> 6), br = row & 63;
      const int pos = S - kBoxRows + br;            // query position of the row
      const bool row_ok = hs < G && br >= kBoxRows - a.r_q;
      float m_run = -INFINITY, l_run = 0.f;
      for (int i = 0; i < n_t; ++i) {
        const int buf = i % n_buf;
        if (!warp_wait(wt, &s_full[buf], (i / n_buf) & 1)) break;
        tc_fence_after();
        const int j0 = (t_begin + i) * a.kt + kh * kw;
        for (int c0 = 0; c0 < kw; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tl + static_cast<uint32_t>(buf) * buf_cols + static_cast<uint32_t>(slot * a.kt + kh * kw + c0), r);
          tmem_wait_ld();
          float v[32];
          float mx = -INFINITY;
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const int j = j0 + c0 + k;
            v[k] = (row_ok && j <= pos) ? __uint_as_float(r[k]) * a.sl2 : -INFINITY;
            mx = fmaxf(mx, v[k]);
          }
          const float m_new = fmaxf(m_run, mx);
          if (m_new != -INFINITY) {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              s0 += ex2(v[k] - m_new);
              s1 += ex2(v[k + 1] - m_new);
            }
            l_run = l_run * ex2(m_run - m_new) + (s0 + s1);
            m_run = m_new;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[buf]);
      }
      if (row_ok && !*abort_flag) {
        const int ir = br - (kBoxRows - a.r_q);
        // one partial per (run, key half): the combine kernel takes n_split * nkh of them
        const size_t o = ((static_cast<size_t>(b) * a.H_kv + g) * a.n_split * nkh + split * nkh + kh) *
                             (G * kBoxRows) + hs * kBoxRows + ir;
        a.part_m[o] = m_run;
        a.part_l[o] = l_run;
      }
    } else {
      // One thread per key of the tile and half of a head's 64 rows (eight warps per
      // head: lane quarter x row half); the tile's heads go in rounds of nph, head
      // hs = round * nph + hp handled by the warps with hp = (e >> 2) & 1.  Per round:
      // the probabilities to shared memory (row br, key jl) and the half column sums;
      // one barrier; the column sums to vsum (the two halves in order) and each thread
      // sums half-diagonals u = br - jl + 127 of the round's heads (a warp reads 32
      // consecutive addresses per row); one barrier before the buffer is written again.
      // The bounded wait for the tile's scores is followed by a barrier and a shared
      // abort check, so the epilogue warps take every barrier together or leave together
      // (only they write epi_abort, and only before that barrier).
      const int nph = static_cast<int>(L.nph);
      const int hp = (e >> 2) & 1, rh = e >> 3;
      const int jl = quarter * 32 + lane;    // key of the tile owned by this thread
      const float *cst = reinterpret_cast<const float *>(sm + L.oC);
      float *P = reinterpret_cast<float *>(sm + L.oP);
      float *s_vs = reinterpret_cast<float *>(sm + L.oV);
      const int n_epi_thr = n_epi * 32;
      const int et = tid - 4 * 32;           // epilogue thread index
      const int n_round = (G + nph - 1) / nph;
      for (int i = 0; i < n_t; ++i) {
        const int buf = i % n_buf;
        const int t = t_begin + i;
        const int j = t * kTile1 + jl;
        if (!warp_wait(wt, &s_full[buf], (i / n_buf) & 1) && lane == 0) *epi_abort = 1;
        named_bar_sync(1, n_epi_thr);
        if (*epi_abort) break;   // the same value for every epilogue warp of this tile
        tc_fence_after();
        for (int rd = 0; rd < n_round; ++rd) {
          const int hs = rd * nph + hp;
          if (hp < nph && hs < G) {
            uint32_t r[32];
            tmem_ld32(tl + static_cast<uint32_t>(buf) * buf_cols + static_cast<uint32_t>(hs * 64 + 32 * rh), r);
            tmem_wait_ld();
            const float4 *c4 = reinterpret_cast<const float4 *>(cst + hs * kBoxRows + 32 * rh);
            float *Ph = P + hp * kBoxRows * kTile1 + 32 * rh * kTile1 + jl;
            // row br attends key j iff br is an estimate row and j <= S - 64 + br
            const int br_lo = max(kBoxRows - a.r_q, j - (S - kBoxRows)) - 32 * rh;
            float vs = 0.f;
#pragma unroll
            for (int b4 = 0; b4 < 8; ++b4) {
              const float4 cc = c4[b4];
              const float cv[4] = {cc.x, cc.y, cc.z, cc.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int br = 4 * b4 + k;
                const float pr = (br >= br_lo && j < S) ? ex2(__uint_as_float(r[br]) * a.sl2 - cv[k]) : 0.f;
                vs += pr;
                Ph[br * kTile1] = pr;
              }
            }
            s_vs[(hp * 2 + rh) * kTile1 + jl] = vs;
          }
          if (rd == n_round - 1) {
            // every score of the tile is in registers: its TMEM buffer is free
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[buf]);
          }
          named_bar_sync(1, n_epi_thr);
          const int n_h = min(nph, G - rd * nph);
          for (int x = et; x < n_h * kTile1; x += n_epi_thr) {
            const int sl = x / kTile1, k = x - sl * kTile1;
            const int jj = t * kTile1 + k;
            if (jj < S)
              a.vsum[(static_cast<size_t>(b) * a.H_q + g * G + rd * nph + sl) * S + jj] =
                  s_vs[(sl * 2) * kTile1 + k] + s_vs[(sl * 2 + 1) * kTile1 + k];
          }
          // one item = one diagonal u of one head, over one half of the rows (two
          // partials per diagonal; the combine kernel adds them)
          for (int x = et; x < n_h * 2 * kDiag1; x += n_epi_thr) {
            const int sl = x / (2 * kDiag1), rem = x - sl * 2 * kDiag1;
            const int half = rem / kDiag1, u = rem - half * kDiag1;
            const float *Ps = P + sl * kBoxRows * kTile1 + (kTile1 - 1) - u + half * 32 * (kTile1 + 1);
            const int lo = max(0, u - (kTile1 - 1)) - 32 * half, hi = min(kBoxRows - 1, u) - 32 * half;
            // all threads walk the same rows in step (predicated outside the diagonal), so
            // the lanes of a warp read consecutive words of one row at a time
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int br = 0; br < 32; br += 2) {
              if (br >= lo && br <= hi) s0 += Ps[br * (kTile1 + 1)];
              if (br + 1 >= lo && br + 1 <= hi) s1 += Ps[(br + 1) * (kTile1 + 1)];
            }
            a.slash_part[(((static_cast<size_t>(b) * a.H_q + g * G + rd * nph + sl) * a.n_ktile + t) * kDiag1 + u) * 2 + half] =
                s0 + s1;
          }
          named_bar_sync(1, n_epi_thr);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    if (lane == 0) drain(fin, 0);   // every MMA retired before TMEM is freed
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && *abort_flag) atomicExch(&g_vs_tc_error, 1);
}

// final row statistics from the runs' partials: one thread per (b, h, estimate row)
__global__ void vs_tc_stats_kernel(const float *part_m, const float *part_l, float *row_m,
                                   float *row_l, int B, int H_q, int H_kv, int r_q, int n_split) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= B * H_q * kBoxRows) return;
  const int i = idx % kBoxRows;
  const int h = (idx / kBoxRows) % H_q;
  const int b = idx / (kBoxRows * H_q);
  if (i >= r_q) return;
  const int G = H_q / H_kv, g = h / G, hs = h - g * G;
  const size_t stride = static_cast<size_t>(G) * kBoxRows;
  const size_t base = (static_cast<size_t>(b) * H_kv + g) * n_split * stride + hs * kBoxRows + i;
  float M = -INFINITY;
  for (int s = 0; s < n_split; ++s) M = fmaxf(M, part_m[base + s * stride]);
  float Ls = 0.f;
  if (M != -INFINITY)
    for (int s = 0; s < n_split; ++s) {
      const float m = part_m[base + s * stride];
      if (m != -INFINITY) Ls += part_l[base + s * stride] * exp2f(m - M);
    }
  row_m[idx] = M;
  row_l[idx] = Ls;
}

// ssum[o] = sum of the pass-1 tile partials of offset o, in ascending tile order
__global__ void vs_slash_tc_kernel(float *ssum, const float *slash_part, int B, int H_q, int S,
                                   int n_ktile, HeadSet heads) {
  const int o = blockIdx.x * blockDim.x + threadIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  if (o >= S || !heads.has(h)) return;
  // tile t covers offsets S - 64 - 128 t - 127 + u, u in [0, 191)
  const int base = S - kBoxRows - (kTile1 - 1) - o;   // = 128 t - u
  int t_lo = base > 0 ? (base + kTile1 - 1) / kTile1 : 0;
  int t_hi = (base + kDiag1 - 1) >= 0 ? (base + kDiag1 - 1) / kTile1 : -1;
  if (t_hi > n_ktile - 1) t_hi = n_ktile - 1;
  const float *sp = slash_part + (static_cast<size_t>(b) * H_q + h) * n_ktile * kDiag1 * 2;
  float s = 0.f;
  for (int t = t_lo; t <= t_hi; ++t) {
    const int u = kTile1 * t - base;
    if (u >= 0 && u < kDiag1) {
      const float2 pr = *reinterpret_cast<const float2 *>(sp + (static_cast<size_t>(t) * kDiag1 + u) * 2);
      s += pr.x + pr.y;
    }
  }
  ssum[(static_cast<size_t>(b) * H_q + h) * S + o] = s;
}

}  // namespace

int vs_tc_tile0(int G) { return G <= 4 ? 128 : 64; }
// warps sharing a row in the row-statistics pass, each on its part of every tile's keys
// (two per row measured slower than one: 142 vs 133 us at 128K)
int vs_tc_khalves(int) { return 1; }
int vs_tc_tile1() { return kTile1; }
int vs_tc_diag() { return 2 * kDiag1; }

void vs_tc_plan(int B, int H_kv, int n_ktile, int *n_split, int *tiles_per_split) {
  // one CTA per SM of a 152-SM part; every split gets at least one tile
  int target = (152 + B * H_kv - 1) / (B * H_kv);
  if (target > n_ktile) target = n_ktile;
  if (target < 1) target = 1;
  const int tps = (n_ktile + target - 1) / target;
  *tiles_per_split = tps;
  *n_split = (n_ktile + tps - 1) / tps;
}

int vs_tc_check(int D, int G) {
  if (D != 64 && D != 128) return fail(DSA_ERR_UNSUPPORTED, "D=%d not in {64, 128}", D);
  if (G < 1 || G > 8) return fail(DSA_ERR_UNSUPPORTED, "H_q/H_kv=%d outside [1, 8]", G);
  return DSA_OK;
}

int vs_tc_ready() {
  if (tensor_map_encoder() == nullptr)
    return fail(DSA_ERR_UNSUPPORTED, "the driver offers no cuTensorMapEncodeTiled entry point");
  return DSA_OK;
}

cudaError_t launch_vs_tc(const VsTcLaunch &l, cudaStream_t s) {
  const int G = l.H_q / l.H_kv;
  const int r_q = l.last_q < l.S ? l.last_q : l.S;
  for (int pass = 0; pass < 2; ++pass) {
    VsTcArgs a;
    std::memset(&a, 0, sizeof(a));
    a.B = l.B;
    a.S = l.S;
    a.H_q = l.H_q;
    a.H_kv = l.H_kv;
    a.G = G;
    a.D = l.D;
    a.r_q = r_q;
    a.kt = pass == 0 ? vs_tc_tile0(G) : kTile1;
    a.n_ktile = (l.S + a.kt - 1) / a.kt;
    vs_tc_plan(l.B, l.H_kv, a.n_ktile, &a.n_split, &a.tiles_per_split);
    a.sl2 = l.scale * kLog2e;
    a.part_m = l.part_m;
    a.part_l = l.part_l;
    a.row_m = l.row_m;
    a.row_l = l.row_l;
    a.vsum = l.vsum;
    a.slash_part = l.slash_part;
    if (!make_bshd_map(&a.tq, l.q, l.D, l.H_q, l.S, l.B, kBoxRows) ||
        !make_bshd_map(&a.tk, l.k, l.D, l.H_kv, l.S, l.B, a.kt))
      return cudaErrorInvalidValue;
    const TcLayout lay(G, l.D, a.kt, pass);
    // at least 116 KB, so that one CTA (and its 512 TMEM columns) holds an SM
    const size_t smem = lay.total + 1024 > 116 * 1024 ? lay.total + 1024 : 116 * 1024;
    const int epi = pass == 0 ? 4 * ((G + 1) / 2) * vs_tc_khalves(G) : 16;
    const int threads = 32 * (4 + epi);
    dim3 grid(a.n_split, l.H_kv, l.B);
    if (pass == 0) {
      auto kern = vs_tc_kernel<0>;
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      ProfScope ps("vs_pass_rowstats", s);
      kern<<<grid, threads, smem, s>>>(a);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      // combine the runs' partials into the final row statistics
      const int total = l.B * l.H_q * kBoxRows;
      ProfScope ps2("vs_combine_rowstats", s);
      vs_tc_stats_kernel<<<(total + 255) / 256, 256, 0, s>>>(l.part_m, l.part_l, l.row_m, l.row_l, l.B,
                                                             l.H_q, l.H_kv, r_q, a.n_split * vs_tc_khalves(G));
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    } else {
      auto kern = vs_tc_kernel<1>;
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      {
        ProfScope ps("vs_pass_sums", s);
        kern<<<grid, threads, smem, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      }
      dim3 g2((l.S + 255) / 256, l.H_q, l.B);
      ProfScope ps("vs_combine_slash", s);
      vs_slash_tc_kernel<<<g2, 256, 0, s>>>(l.ssum, l.slash_part, l.B, l.H_q, l.S, a.n_ktile, l.heads);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

int vs_tc_set_wait_limit(unsigned long long ns) {
  return cudaMemcpyToSymbol(g_vs_wait_limit_ns, &ns, sizeof(ns)) == cudaSuccess ? 0 : -1;
}

int vs_tc_device_error() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_vs_tc_error, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_vs_tc_error, &zero, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

}  // namespace dsa
