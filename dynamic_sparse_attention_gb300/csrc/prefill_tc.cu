// Sparse causal prefill attention on sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// Source: "MInference 1.0: Accelerating Pre-filling for Long-Context LLMs via Dynamic
// Sparse Attention" (paper-graph-ui summary): "Vertical-Slash Hybrid Kernel" (Alg. 5:
// block phase over 64x64 tiles, then gathered column tiles, one online softmax) and
// "Block-Sparse FlashAttention Kernel (Appendix C.4.1)"; section 3.4 Eq. 1 with the
// mask constant taken as exact exclusion.
//
// One CTA computes 128 query rows: the two consecutive 64-row query blocks m0 = 2p and
// m1 = 2p + 1 of one head, so every MMA has M = 128.  The CTA walks the union of the two
// blocks' tile lists (ascending key block), then block m0's column tiles, then block
// m1's; a tile listed for only one of the blocks is masked for the other half's rows.
// Warp roles (192 threads):
//   warp 0    producer: Q once (TMA), then per tile K and V (TMA for 64-key blocks,
//             16-byte cp.async gathers for column tiles) into a 4-stage ring;
//   warp 1    MMA issuer (one thread): S = Q K^T into a double-buffered TMEM tile
//             (128 lanes x 64 fp32 columns), O += P V into TMEM (128 x D fp32);
//   warps 2-5 softmax, one thread per query row: read S from TMEM, mask, online
//             softmax with the exact running max (when a row's max grows, O in TMEM
//             is rescaled once the previous P V has retired, so the largest
//             probability of a row is exactly 1 and carries no bf16 rounding), write
//             P (bf16) to shared memory in the 128-byte-swizzled K-major layout the
//             MMA reads, and at the end normalise O and store it.
// Operands: Q and K tiles are K-major with 128-byte swizzle (what TMA writes for a
// 64-element-wide box); V tiles are the B operand in MN-major form (keys along K).
// Every mbarrier wait is bounded; on a timeout the CTA stops issuing work, drains its
// copies and MMAs, frees TMEM, records an error word and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "api_common.h"
#include "common.cuh"
#include "launch.h"
#include "mma_sync.cuh"
#include "profile.h"
#include "tc_ptx.cuh"

namespace dsa {
namespace {

using namespace tc;

constexpr int kRowsQ = 128;       // query rows per CTA
constexpr int kKeys = 64;         // keys per tile
constexpr int kNS = 4;            // K/V pipeline stages
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

static __device__ int g_prefill_tc_error;   // sticky error word, read by dsa_device_error
static __device__ int g_abort_epoch;         // launch epoch of a launch in which a CTA gave up
constexpr uint64_t kWaitLimitNs = 500000000ull;

struct TileMeta {
  int kind;          // 0: 64-key block, 1: gathered column tile
  int n;             // key block (kind 0)
  int mask;          // bit 0: rows of block m0 use the tile, bit 1: rows of block m1
  int ncols;
  int pos[kKeys];    // key positions of a column tile (-1: empty slot)
};

template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kQHalf = kRowsQ * 128;          // 128 rows x 128 bytes
  static constexpr uint32_t kKVHalf = kKeys * 128;          // 64 rows x 128 bytes
  static constexpr uint32_t kStage = 2 * kHalves * kKVHalf;   // K halves, then V halves
  static constexpr uint32_t kP = kRowsQ * 128;              // 128 rows x 64 bf16
  static constexpr uint32_t oQ = 0;
  static constexpr uint32_t oStage = oQ + kHalves * kQHalf;
  static constexpr uint32_t oP = oStage + kNS * kStage;
  static constexpr uint32_t oMeta = oP + 2 * kP;
  static constexpr uint32_t oBar = oMeta + kNS * sizeof(TileMeta);
  static constexpr int kBars = 2 * kNS + 8;
  static constexpr uint32_t oMisc = oBar + kBars * 8;
  static constexpr uint32_t oBits = oMisc + 64;
  static size_t bytes(int n_words) { return oBits + 8ull * n_words + 1024; }
};

struct TcArgs {
  CUtensorMap tq, tk, tv;
  const uint16_t *k, *v;
  const int32_t *blk_cnt, *blk_idx, *col_cnt, *col_idx;
  uint16_t *out;
  float *lse;
  int B, S, H_q, H_kv, max_blk, max_col, n_qblk, n_words;
  float sl2;
  int epoch;   // distinct per launch
};

struct WaitCtx {
  volatile int *cta_abort;
  int epoch;
};

// Bounded mbarrier wait.  Gives up when this CTA already gave up, when another CTA of
// the same launch gave up (epoch word), or after kWaitLimitNs; returns false then.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, const WaitCtx &w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*w.cta_abort) return false;
    if ((++spins & 31u) == 0u) {
      if (*reinterpret_cast<volatile int *>(&g_abort_epoch) == w.epoch) {
        *w.cta_abort = 1;
        return false;
      }
      if (global_ns() - t0 > kWaitLimitNs) {
        *w.cta_abort = 1;
        atomicExch(&g_abort_epoch, w.epoch);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) return false;
  return true;
}

// lane 0 waits, the warp learns the outcome (keeps tcgen05 collectives warp-uniform)
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const WaitCtx &w) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = tc_wait(bar, parity, w) ? 1 : 0;
  ok = __shfl_sync(kFull, ok, 0);
  __syncwarp();
  return ok != 0;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcArgs a) {
  using L = Layout<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::oBar);
  uint64_t *kv_full = bars, *kv_empty = bars + kNS;
  uint64_t *s_full = bars + 2 * kNS, *p_full = s_full + 2, *pv_done = p_full + 2;
  uint64_t *q_full = pv_done + 2, *fin = q_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::oMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::oMisc + 4);
  int *n_blk_tiles_s = reinterpret_cast<int *>(sm + L::oMisc + 8);
  uint32_t *bm0 = reinterpret_cast<uint32_t *>(sm + L::oBits);
  uint32_t *bm1 = bm0 + a.n_words;
  TileMeta *meta = reinterpret_cast<TileMeta *>(sm + L::oMeta);
  const WaitCtx wc{abort_flag, a.epoch};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_pairs = (a.n_qblk + 1) / 2;
  const int p = n_pairs - 1 - static_cast<int>(blockIdx.x);
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (a.H_q / a.H_kv);
  const int m0 = 2 * p, m1 = 2 * p + 1;
  const bool has1 = m1 < a.n_qblk;
  const size_t bh = static_cast<size_t>(b) * a.H_q + h;

  if (tid == 0) {
    for (int i = 0; i < 2 * kNS; ++i) mbar_init(&bars[i], 1);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&p_full[0], 128);
    mbar_init(&p_full[1], 128);
    mbar_init(&pv_done[0], 1);
    mbar_init(&pv_done[1], 1);
    mbar_init(q_full, 1);
    mbar_init(fin, 1);
    *abort_flag = 0;
    *n_blk_tiles_s = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  for (int w = tid; w < 2 * a.n_words; w += kThreads) bm0[w] = 0u;
  __syncthreads();
  // tile lists -> bitmaps; a block after a half's own query block is fully masked there
  {
    const int c = min(max(a.blk_cnt[bh * a.n_qblk + m0], 0), a.max_blk);
    const int32_t *l0 = a.blk_idx + (bh * a.n_qblk + m0) * static_cast<size_t>(a.max_blk);
    for (int i = tid; i < c; i += kThreads) {
      const int n = l0[i];
      if (n >= 0 && n <= m0) atomicOr(&bm0[n >> 5], 1u << (n & 31));
    }
    if (has1) {
      const int c1 = min(max(a.blk_cnt[bh * a.n_qblk + m1], 0), a.max_blk);
      const int32_t *l1 = a.blk_idx + (bh * a.n_qblk + m1) * static_cast<size_t>(a.max_blk);
      for (int i = tid; i < c1; i += kThreads) {
        const int n = l1[i];
        if (n >= 0 && n <= m1) atomicOr(&bm1[n >> 5], 1u << (n & 31));
      }
    }
  }
  __syncthreads();
  {
    int cnt = 0;
    for (int w = tid; w < a.n_words; w += kThreads) cnt += __popc(bm0[w] | bm1[w]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(kFull, cnt, o);
    if (lane == 0 && cnt) atomicAdd(n_blk_tiles_s, cnt);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int n_blk_t = *n_blk_tiles_s;
  const int c0 = min(max(a.col_cnt[bh * a.n_qblk + m0], 0), a.max_col);
  const int c1 = has1 ? min(max(a.col_cnt[bh * a.n_qblk + m1], 0), a.max_col) : 0;
  const int nct0 = (c0 + kKeys - 1) / kKeys, nct1 = (c1 + kKeys - 1) / kKeys;
  const int T = n_blk_t + nct0 + nct1;
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, L::kHalves * L::kQHalf);
      for (int hh = 0; hh < L::kHalves; ++hh)
        tma_load_4d(sm + L::oQ + hh * L::kQHalf, &a.tq, q_full, 64 * hh, h, kRowsQ * p, b);
    }
    int wi = 0;
    uint32_t cur = a.n_words > 0 ? (bm0[0] | bm1[0]) : 0u;
    int issued = 0;
    const size_t krow = static_cast<size_t>(a.H_kv) * D;
    const uint16_t *kb = a.k + (static_cast<size_t>(b) * a.S * a.H_kv + g) * D;
    const uint16_t *vb = a.v + (static_cast<size_t>(b) * a.S * a.H_kv + g) * D;
    for (int t = 0; t < T; ++t) {
      const int st = t % kNS;
      if (t >= kNS && !warp_wait(&kv_empty[st], ((t / kNS) - 1) & 1, wc)) break;
      unsigned char *stage = sm + L::oStage + st * L::kStage;
      TileMeta *md = &meta[st];
      if (t < n_blk_t) {
        if (lane == 0 && cur == 0u) {
          while (cur == 0u && wi + 1 < a.n_words) {
            ++wi;
            cur = bm0[wi] | bm1[wi];
          }
          if (cur == 0u) *abort_flag = 1;   // count and bitmaps disagree: stop cleanly
        }
        if (__shfl_sync(kFull, static_cast<int>(*abort_flag), 0)) break;
        if (lane == 0) {
          const int n = wi * 32 + __ffs(cur) - 1;
          cur &= cur - 1u;
          md->kind = 0;
          md->n = n;
          md->mask = ((bm0[n >> 5] >> (n & 31)) & 1u) | (((bm1[n >> 5] >> (n & 31)) & 1u) << 1);
          md->ncols = kKeys;
          mbar_arrive_expect_tx(&kv_full[st], L::kStage);
          for (int hh = 0; hh < L::kHalves; ++hh)
            tma_load_4d(stage + hh * L::kKVHalf, &a.tk, &kv_full[st], 64 * hh, g, kKeys * n, b);
          for (int hh = 0; hh < L::kHalves; ++hh)
            tma_load_4d(stage + (L::kHalves + hh) * L::kKVHalf, &a.tv, &kv_full[st], 64 * hh, g,
                        kKeys * n, b);
        }
      } else {
        const int ct = t - n_blk_t;
        const int grp = ct < nct0 ? 0 : 1;
        const int cb = (grp == 0 ? ct : ct - nct0) * kKeys;
        const int mg = grp == 0 ? m0 : m1;
        const int cg = grp == 0 ? c0 : c1;
        const int32_t *cl = a.col_idx + (bh * a.n_qblk + mg) * static_cast<size_t>(a.max_col);
        const int ncol = min(kKeys, cg - cb);
        const int last_row = min(kKeys * mg + kKeys - 1, a.S - 1);
        for (int x = lane; x < kKeys; x += 32) {
          int j = x < ncol ? cl[cb + x] : -1;
          if (j < 0 || j > last_row) j = -1;
          md->pos[x] = j;
        }
        if (lane == 0) {
          md->kind = 1;
          md->n = -1;
          md->mask = 1 << grp;
          md->ncols = ncol;
        }
        __syncwarp();
        constexpr int CPR = D / 8;   // 16-byte chunks per row
        for (int e = lane; e < 2 * kKeys * CPR; e += 32) {
          const int which = e / (kKeys * CPR);
          const int rem = e - which * (kKeys * CPR);
          const int x = rem / CPR, c = rem - x * CPR;
          const int hh = c >> 3, cc = c & 7;
          unsigned char *dst = stage + (which * L::kHalves + hh) * L::kKVHalf + x * 128 +
                               ((cc ^ (x & 7)) << 4);
          const int j = md->pos[x];
          if (j >= 0) cp_async_16(dst, (which ? vb : kb) + static_cast<size_t>(j) * krow + c * 8);
          else *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
        }
        cp_async_wait<0>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&kv_full[st]);
      }
      ++issued;
    }
    if (*abort_flag && lane == 0) {
      // let this CTA's copies land before it exits
      for (int t = max(0, issued - kNS); t < issued; ++t)
        drain_wait(&kv_full[t % kNS], (t / kNS) & 1, 200000000ull);
      drain_wait(q_full, 0, 200000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16_f32(kRowsQ, kKeys, false, false);
      constexpr uint32_t id_pv = idesc_bf16_f32(kRowsQ, D, false, true);
      const uint32_t sQ = smem_u32(sm + L::oQ);
      const uint32_t sS = smem_u32(sm + L::oStage);
      const uint32_t sP = smem_u32(sm + L::oP);
      bool ok = tc_wait(q_full, 0, wc);
      auto issue_qk = [&](int t) -> bool {
        const int st = t % kNS;
        if (!tc_wait(&kv_full[st], (t / kNS) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>((t & 1) * kKeys);
        const uint32_t kbase = sS + st * L::kStage;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(sQ + (kk >> 2) * L::kQHalf + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(kbase + (kk >> 2) * L::kKVHalf + (kk & 3) * 32, 16, 1024);
          tc_mma(d, ad, bd, id_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[t & 1]);
        return true;
      };
      if (ok && T > 0) ok = issue_qk(0);
      for (int t = 0; ok && t < T; ++t) {
        if (t + 1 < T && !(ok = issue_qk(t + 1))) break;
        if (!(ok = tc_wait(&p_full[t & 1], (t >> 1) & 1, wc))) break;
        tc_fence_after();
        const uint32_t vbase = sS + (t % kNS) * L::kStage + L::kHalves * L::kKVHalf;
        const uint32_t pbase = sP + (t & 1) * L::kP;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(pbase + kk * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(vbase + kk * 2048, L::kKVHalf, 1024);
          tc_mma(tmem + 2 * kKeys, ad, bd, id_pv, (t > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&pv_done[t & 1]);
        tc_commit(&kv_empty[t % kNS]);
      }
      tc_commit(fin);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int grp = row >> 6;
    const int qpos = kRowsQ * p + row;
    const bool row_ok = qpos < a.S;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int sb = t & 1;
      if (!(ok = warp_wait(&s_full[sb], (t >> 1) & 1, wc))) break;
      tc_fence_after();
      uint32_t sr[2 * 32];
      tmem_ld32(tl + sb * kKeys, sr);
      tmem_ld32(tl + sb * kKeys + 32, sr + 32);
      tmem_wait_ld();
      const TileMeta *md = &meta[t % kNS];
      const int kind = md->kind;
      const bool member = row_ok && ((md->mask >> grp) & 1);
      float mt = -INFINITY;
      if (!member) {
#pragma unroll
        for (int c = 0; c < kKeys; ++c) sr[c] = __float_as_uint(-INFINITY);
      } else if (kind == 0) {
        const int lim = min(qpos, a.S - 1) - kKeys * md->n;   // slots 0..lim are keys <= row
        if (lim >= kKeys - 1) {
#pragma unroll
          for (int c = 0; c < kKeys; ++c) {
            const float x = __uint_as_float(sr[c]) * a.sl2;
            sr[c] = __float_as_uint(x);
            mt = fmaxf(mt, x);
          }
        } else {
#pragma unroll
          for (int c = 0; c < kKeys; ++c) {
            const float x = c <= lim ? __uint_as_float(sr[c]) * a.sl2 : -INFINITY;
            sr[c] = __float_as_uint(x);
            mt = fmaxf(mt, x);
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < kKeys; ++c) {
          const int j = md->pos[c];
          const float x = (j >= 0 && j <= qpos) ? __uint_as_float(sr[c]) * a.sl2 : -INFINITY;
          sr[c] = __float_as_uint(x);
          mt = fmaxf(mt, x);
        }
      }
      const bool resc = m_ref != -INFINITY && mt > m_ref;
      if (__any_sync(kFull, resc)) {
        // O holds PV_{t-1}'s result only after it completes
        if (t >= 1 && !(ok = warp_wait(&pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, wc))) break;
        tc_fence_after();
        const float f = resc ? exp2f(m_ref - mt) : 1.f;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(tl + 2 * kKeys + ch * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
          tmem_st32(tl + 2 * kKeys + ch * 32, o);
        }
        tmem_wait_st();
        if (resc) {
          l *= f;
          m_ref = mt;
        }
      }
      if (m_ref == -INFINITY) m_ref = mt;
      uint32_t pk[kKeys / 2];
      float ps = 0.f;
#pragma unroll
      for (int c = 0; c < kKeys; c += 2) {
        float p0 = 0.f, p1 = 0.f;
        if (m_ref != -INFINITY) {
          p0 = fast_exp2(__uint_as_float(sr[c]) - m_ref);
          p1 = fast_exp2(__uint_as_float(sr[c + 1]) - m_ref);
        }
        ps += p0 + p1;
        pk[c >> 1] = pack_bf16x2(p0, p1);
      }
      l += ps;
      // the P buffer is free once PV_{t-2} has completed
      if (t >= 2 && !(ok = warp_wait(&pv_done[sb], ((t - 2) >> 1) & 1, wc))) break;
      unsigned char *prow = sm + L::oP + sb * L::kP + row * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4 *>(prow + ((c ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[sb]);
    }
    const bool have_o = ok && T > 0 && warp_wait(&pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1, wc);
    if (have_o) tc_fence_after();
    const float inv = (have_o && l > 0.f) ? 1.f / l : 0.f;
    uint16_t *orow = a.out + ((static_cast<size_t>(b) * a.S + (row_ok ? qpos : 0)) * a.H_q + h) * D;
#pragma unroll 1
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t o[32];
      if (have_o) {
        tmem_ld32(tl + 2 * kKeys + ch * 32, o);
        tmem_wait_ld();
      }
      if (row_ok) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = have_o ? pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv)
                        : 0u;
        uint4 *dst = reinterpret_cast<uint4 *>(orow + ch * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      }
    }
    if (row_ok && a.lse)
      a.lse[bh * a.S + qpos] = (have_o && l > 0.f) ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if (lane == 0) drain_wait(fin, 0, 1000000000ull);   // every MMA retired before TMEM is freed
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && *abort_flag) atomicExch(&g_prefill_tc_error, 1);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 4-D view (d, head, position, batch) of a bshd bf16 tensor; box = 64 d x 1 x rows x 1
bool make_map(CUtensorMap *m, const void *base, int D, int H, int S, int B, int rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                           static_cast<cuuint64_t>(S) * H * D * 2};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(rows), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_tc_d(const PrefillArgs &pa, cudaStream_t s) {
  TcArgs a;
  std::memset(&a, 0, sizeof(a));
  if (!make_map(&a.tq, pa.q, D, pa.H_q, pa.S, pa.B, kRowsQ) ||
      !make_map(&a.tk, pa.k, D, pa.H_kv, pa.S, pa.B, kKeys) ||
      !make_map(&a.tv, pa.v, D, pa.H_kv, pa.S, pa.B, kKeys))
    return cudaErrorInvalidValue;
  a.k = static_cast<const uint16_t *>(pa.k);
  a.v = static_cast<const uint16_t *>(pa.v);
  a.blk_cnt = pa.blk_cnt;
  a.blk_idx = pa.blk_idx;
  a.col_cnt = pa.col_cnt;
  a.col_idx = pa.col_idx;
  a.out = static_cast<uint16_t *>(pa.out);
  a.lse = pa.lse;
  a.B = pa.B;
  a.S = pa.S;
  a.H_q = pa.H_q;
  a.H_kv = pa.H_kv;
  a.max_blk = pa.max_blk;
  a.max_col = pa.max_col;
  a.n_qblk = (pa.S + 63) / 64;
  a.n_words = (a.n_qblk + 31) / 32;
  a.sl2 = pa.scale * kLog2e;
  static std::atomic<int> epoch{0};
  int ep = ++epoch;
  if (ep <= 0) ep = epoch = 1;
  a.epoch = ep;
  const size_t smem = Layout<D>::bytes(a.n_words);
  auto kern = prefill_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.n_qblk + 1) / 2, pa.H_q, pa.B);
  {
    ProfScope ps("prefill_attention_tc", s);
    kern<<<grid, kThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs &a) {
  if (a.D != 64 && a.D != 128) return false;
  const int n_qblk = (a.S + 63) / 64;
  const size_t smem = a.D == 128 ? Layout<128>::bytes((n_qblk + 31) / 32)
                                 : Layout<64>::bytes((n_qblk + 31) / 32);
  return smem <= 227 * 1024 && encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t s) {
  return a.D == 128 ? launch_tc_d<128>(a, s) : launch_tc_d<64>(a, s);
}

}  // namespace dsa

extern "C" int dsa_device_error(int *code) {
  using namespace dsa;
  clear_error();
  if (!code) return fail(DSA_ERR_ALIGNMENT, "code is NULL");
  int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_prefill_tc_error, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_prefill_tc_error, &zero, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  *code = v;
  return DSA_OK;
}
