// Sparse causal prefill attention on sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// Source: "MInference 1.0: Accelerating Pre-filling for Long-Context LLMs via Dynamic
// Sparse Attention" (paper-graph-ui summary): "Vertical-Slash Hybrid Kernel" (Alg. 5:
// block phase over 64x64 tiles, then gathered column tiles, one online softmax) and
// "Block-Sparse FlashAttention Kernel (Appendix C.4.1)"; section 3.4 Eq. 1 with the
// mask constant taken as exact exclusion.
//
// One CTA computes 128 query rows in two 64-row groups: the consecutive query blocks
// m0 = 2p and m1 = 2p + 1 of one head, or, where two query heads of one KV head list
// the same blocks and columns for both blocks of the pair, one query block of both
// heads (the two CTAs of such a head pair split the pair's blocks between them).  Keys
// go through the tensor core in 128-key tiles, each made of two 64-key list blocks: at
// M = N = K = 128 the MMA runs at its full rate, while 64-key tiles (Q K^T with N = 64,
// P V with K = 64) reach well under half of it.  The CTA walks the blocks that either
// group lists (the union of the two lists), in descending order, and puts each next two
// of them into a tile (descending, so the running max settles early; any two blocks, so
// scattered lists fill their tiles), then group 0's gathered column tiles (128 columns
// each), then group 1's (none when both groups share the columns: one walk serves
// both).  A row masks the 64-key halves its own group does not list, keys after it
// (causal) and keys past the sequence end.
// Warp roles (352 threads):
//   warp 0     K producer: Q once (TMA), then K tiles (two 64-row TMA boxes per 64-wide
//              head-dim half for block tiles, 16-byte cp.async gathers for column tiles,
//              which complete on the stage's mbarrier while the warp moves on) into a
//              3-stage ring; writes each tile's description (kind, the block of each
//              half, per-half membership, column positions);
//   warp 1     V producer: V tiles into a 2-stage ring (its own walk of the same lists);
//   warp 2     MMA issuer (one thread): S_b = Q K^T (M = N = 128, K = D) into one of three
//              TMEM score buffers (b = tile mod 3), O += P V (A = P read from TMEM,
//              128 keys).  Q K^T of tile t + 3 is queued right behind P V of tile t, so
//              the scores of the next two tiles are ready while tile t is in softmax;
//   warps 3-10 softmax: two threads per query row; warp w reads the TMEM lanes of
//              quarter w % 4 and the 64-key half w / 4 of the tile.  The two halves of a
//              row exchange their maxima through shared memory (an mbarrier per lane
//              quarter); each thread then forms P = exp2(s * scale * log2e - m) against
//              a reference m that follows the running max lazily: it moves to the max
//              only once the max exceeds it by more than kRescaleSlack (so P <= 2),
//              keeps a partial row sum, and writes its bf16 pairs over the first 64
//              columns of S_b, where the P V MMA reads them, while the next tile's scores
//              stream in from TMEM.  When the reference moves, each warp brings its
//              quarter of O to it once P V of the previous tile has retired (a wait that
//              drains the MMA pipe, hence the slack).  The epilogue adds the partial
//              sums, normalises and stores.
// Operands: Q and K tiles are K-major with 128-byte swizzle (what TMA writes for a
// 64-element-wide box); V tiles are the B operand in MN-major form (keys along K).
// Every mbarrier wait is bounded; on a timeout the CTA stops issuing work, drains its
// copies and MMAs, frees TMEM, records an error word and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <atomic>
#include <cstdlib>
#include <cstddef>
#include <cstring>
#include <mutex>

#include "api_common.h"
#include "common.cuh"
#include "launch.h"
#include "mma_sync.cuh"
#include "profile.h"
#include "tc_ptx.cuh"

namespace dsa {

DSA_CHECK_WORD(prefill_tc_check_word)

namespace {

using namespace tc;

constexpr int kRowsQ = 128;        // query rows per CTA
constexpr int kBlk = 64;           // block size of the tile lists
constexpr int kKeys = 128;         // keys per MMA tile (two list blocks, one per 64-key half)
constexpr int kKS = 3;             // K ring stages
constexpr int kVS = 2;             // V ring stages
constexpr int kSB = 3;             // TMEM score buffers
constexpr int kMetaRing = 8;       // tile descriptions in flight (the K ring runs at most 6 ahead)
constexpr int kSlices = 2;         // key slices per query row (threads per row)
constexpr int kSW = kKeys / kSlices;   // keys per slice
constexpr int kSmWarps = 4 * kSlices;  // softmax warps: 4 TMEM lane quarters x kSlices
constexpr int kThreads = (3 + kSmWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// log2 units by which a row's max may exceed its softmax reference before the
// reference (and O with it) is moved.  With 1, P <= 2 and the bf16 rounding of the
// probabilities is that of the exact-max form (measured on the parity cases: the same
// worst error; 2 and 4 raise it, 4 past the 1e-2 bound), while most of the rescales,
// each a wait on the previous P V by every warp with a row whose max moved, go away.
constexpr float kRescaleSlack = 1.f;

static __device__ int g_prefill_tc_error;   // sticky error word, read by dsa_device_error
static __device__ int g_abort_epoch;         // launch epoch of a launch in which a CTA gave up
constexpr uint64_t kWaitLimitNs = 500000000ull;
// wait limit of the kernel's bounded waits (dsa_set_wait_limit; default kWaitLimitNs)
static __device__ unsigned long long g_wait_limit_ns = kWaitLimitNs;

struct TileMeta {
  int kind;          // 0: block tile (two 64-key list blocks), 1: gathered column tile
  int mask;          // bit 2*grp + half: rows of query block m_grp use that 64-key half
  int blk[2];        // the 64-key block held by each half (kind 0)
  int below;         // kind 1: every key precedes every row of the tile's query block
  int pad[3];
  uint32_t nonempty[kKeys / 32];   // kind 1: bit x: slot x holds a key
  int pos[kKeys];    // key positions of a column tile (-1: empty slot)
};
static_assert(sizeof(TileMeta) % 16 == 0 && offsetof(TileMeta, pos) % 16 == 0, "int4 reads of pos");

template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kQHalf = kRowsQ * 128;          // 128 rows x 64 dims
  static constexpr uint32_t kHalf = kKeys * 128;            // 128 keys x 64 dims
  static constexpr uint32_t kTile = kHalves * kHalf;        // one K or V tile
  static constexpr uint32_t oQ = 0;
  static constexpr uint32_t oK = oQ + kHalves * kQHalf;
  static constexpr uint32_t oV = oK + kKS * kTile;
  static constexpr uint32_t oMeta = oV + kVS * kTile;
  static constexpr uint32_t oBar = oMeta + kMetaRing * sizeof(TileMeta);
  // rings, score buffers, q_full, fin, then per lane quarter: max exchange x2, sum exchange
  static constexpr int kBars = 2 * kKS + 2 * kVS + 3 * kSB + 2 + 4 * 3;
  static constexpr uint32_t oMisc = oBar + kBars * 8;
  static constexpr uint32_t oRed = oMisc + 64;              // [3][kSlices][128 rows] floats
  static constexpr uint32_t oBits = oRed + 3 * kSlices * kRowsQ * 4;
  static size_t bytes(int n_words) { return oBits + 8ull * n_words + 1024; }
  // TMEM columns (32-bit): S_0, S_1, S_2 (P_b over the first 64 columns of S_b) | O
  static constexpr uint32_t cO = kSB * kKeys;
  static_assert(cO + D <= kTmemCols, "TMEM columns");
  static_assert(oQ % 1024 == 0 && oK % 1024 == 0 && oV % 1024 == 0, "swizzle atoms");
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
  const uint64_t limit = g_wait_limit_ns;
  const uint32_t hint = limit < 20000ull ? static_cast<uint32_t>(limit) : 20000u;
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait_hint(bar, parity, hint)) return true;
    if (*w.cta_abort) return false;
    if ((++spins & 7u) == 0u) {
      if (*reinterpret_cast<volatile int *>(&g_abort_epoch) == w.epoch) {
        *w.cta_abort = 1;
        return false;
      }
      if (global_ns() - t0 > limit) {
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

// Walk over the blocks either query block lists, in descending key order, two per
// tile (run by one lane).  Scores near the diagonal are usually the largest of a row,
// so visiting them first settles the running max early and spares most rescalings of
// the accumulator.
struct TileWalk {
  const uint32_t *bm0, *bm1;
  int wi;
  uint32_t cur;
  __device__ void init(const uint32_t *b0, const uint32_t *b1, int nw) {
    bm0 = b0;
    bm1 = b1;
    wi = nw - 1;
    cur = nw > 0 ? (bm0[wi] | bm1[wi]) : 0u;
  }
  __device__ bool next_block(int &j) {
    while (cur == 0u && wi > 0) {
      --wi;
      cur = bm0[wi] | bm1[wi];
    }
    if (cur == 0u) return false;
    const int bit = 31 - __clz(cur);
    cur &= ~(1u << bit);
    j = wi * 32 + bit;
    return true;
  }
  // next tile: its two blocks (an odd last block is loaded twice, its second half
  // unused) and its membership mask; false once the bitmaps run out
  __device__ bool next(int &ja, int &jb, int &mask) {
    if (!next_block(ja)) return false;
    const bool two = next_block(jb);
    if (!two) jb = ja;
    auto in = [](const uint32_t *bm, int j) { return static_cast<int>((bm[j >> 5] >> (j & 31)) & 1u); };
    mask = in(bm0, ja) | ((two ? in(bm0, jb) : 0) << 1) | (in(bm1, ja) << 2) |
           ((two ? in(bm1, jb) : 0) << 3);
    return true;
  }
};

// The CTA's work once its row groups are chosen (HP: two query heads of one query block,
// else two query blocks of one query head): list bitmaps, then the warp roles.  Both
// forms are compiled separately so that each keeps the code of a fixed row layout.
template <int D, bool HP>
__device__ __forceinline__ void tc_cta(const TcArgs &a, unsigned char *sm, int p, int g, int b, int hl,
                                       int hA) {
  using L = Layout<D>;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::oBar);
  uint64_t *k_full = bars, *k_empty = k_full + kKS;
  uint64_t *v_full = k_empty + kKS, *v_empty = v_full + kVS;
  uint64_t *s_full = v_empty + kVS, *p_full = s_full + kSB;
  uint64_t *pv_done = p_full + kSB, *q_full = pv_done + kSB, *fin = q_full + 1;
  uint64_t *xbar = fin + 1;   // [4 quarters][3]: row-max exchange by tile parity, row sums
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::oMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::oMisc + 4);
  int *n_blk_tiles_s = reinterpret_cast<int *>(sm + L::oMisc + 8);
  uint32_t *bm0 = reinterpret_cast<uint32_t *>(sm + L::oBits);
  uint32_t *bm1 = bm0 + a.n_words;
  TileMeta *meta = reinterpret_cast<TileMeta *>(sm + L::oMeta);
  const WaitCtx wc{abort_flag, a.epoch};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.H_q / a.H_kv;
  // the two row groups: query head and query block of each, and their list rows
  const int hq0 = HP ? hA : g * G + hl, hq1 = HP ? hA + 1 : hq0;
  const int m0 = HP ? 2 * p + (hl & 1) : 2 * p, m1 = HP ? m0 : 2 * p + 1;
  const bool has1 = m1 < a.n_qblk;
  const size_t lr0 = (static_cast<size_t>(b) * a.H_q + hq0) * a.n_qblk + m0;
  const size_t lr1 = (static_cast<size_t>(b) * a.H_q + hq1) * a.n_qblk + m1;
  // tile lists -> bitmaps; a block after a half's own query block is fully masked there
  {
    const int c_raw = a.blk_cnt[lr0];
    DSA_CHECK(c_raw >= 0 && c_raw <= a.max_blk);
    const int c = min(max(c_raw, 0), a.max_blk);
    const int32_t *l0 = a.blk_idx + lr0 * static_cast<size_t>(a.max_blk);
    for (int i = tid; i < c; i += kThreads) {
      const int n = l0[i];
      DSA_CHECK(n >= 0 && n < a.n_qblk);
      if (n >= 0 && n <= m0) atomicOr(&bm0[n >> 5], 1u << (n & 31));
    }
    if (has1) {
      const int c1_raw = a.blk_cnt[lr1];
      DSA_CHECK(c1_raw >= 0 && c1_raw <= a.max_blk);
      const int c1 = min(max(c1_raw, 0), a.max_blk);
      const int32_t *l1 = a.blk_idx + lr1 * static_cast<size_t>(a.max_blk);
      for (int i = tid; i < c1; i += kThreads) {
        const int n = l1[i];
        DSA_CHECK(n >= 0 && n < a.n_qblk);
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
  const int n_blk_t = (*n_blk_tiles_s + 1) / 2;   // listed blocks, two per tile
  const int cc0_raw = a.col_cnt[lr0];
  const int cc1_raw = has1 ? a.col_cnt[lr1] : 0;
  DSA_CHECK(cc0_raw >= 0 && cc0_raw <= a.max_col && cc1_raw >= 0 && cc1_raw <= a.max_col);
  const int c0 = min(max(cc0_raw, 0), a.max_col);
  const int c1 = has1 ? min(max(cc1_raw, 0), a.max_col) : 0;
  // one column walk for both groups when they list the same columns (head pairs)
  const int nct0 = (c0 + kKeys - 1) / kKeys, nct1 = HP ? 0 : (c1 + kKeys - 1) / kKeys;
  const int T = n_blk_t + nct0 + nct1;
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 || warp == 1) {
    // ------------------------------------------------------------ producers (K: warp 0, V: warp 1)
    const bool is_k = warp == 0;
    const int NS = is_k ? kKS : kVS;
    uint64_t *full = is_k ? k_full : v_full;
    uint64_t *empty = is_k ? k_empty : v_empty;
    unsigned char *ring = sm + (is_k ? L::oK : L::oV);
    const CUtensorMap *map = is_k ? &a.tk : &a.tv;
    const uint16_t *src = (is_k ? a.k : a.v) + (static_cast<size_t>(b) * a.S * a.H_kv + g) * D;
    const size_t krow = static_cast<size_t>(a.H_kv) * D;
    if (is_k && lane == 0) {
      // Q rows 0-63 from (hq0, block m0), 64-127 from (hq1, block m1), per head-dim half
      mbar_arrive_expect_tx(q_full, L::kHalves * L::kQHalf);
      for (int hh = 0; hh < L::kHalves; ++hh) {
        tma_load_4d(sm + L::oQ + hh * L::kQHalf, &a.tq, q_full, 64 * hh, hq0, kBlk * m0, b);
        tma_load_4d(sm + L::oQ + hh * L::kQHalf + L::kQHalf / 2, &a.tq, q_full, 64 * hh, hq1, kBlk * m1, b);
      }
    }
    TileWalk walk;
    walk.init(bm0, bm1, a.n_words);
    int issued = 0;
    for (int t = 0; t < T; ++t) {
      const int st = t % NS;
      if (t >= NS && !warp_wait(&empty[st], ((t / NS) - 1) & 1, wc)) break;
      unsigned char *stage = ring + st * L::kTile;
      if (t < n_blk_t) {
        int ja = 0, jb = 0, mask = 0, ok = 1;
        if (lane == 0) {
          ok = walk.next(ja, jb, mask) ? 1 : 0;
          if (!ok) *abort_flag = 1;   // count and bitmaps disagree: stop cleanly
        }
        if (!__shfl_sync(kFull, ok, 0)) break;
        if (lane == 0) {
          if (is_k) {
            TileMeta *md = &meta[t % kMetaRing];
            md->kind = 0;
            md->mask = mask;
            md->blk[0] = ja;
            md->blk[1] = jb;
          }
          // rows 0-63 of the tile from block ja, rows 64-127 from block jb, per head-dim half
          mbar_arrive_expect_tx(&full[st], L::kTile);
          for (int hh = 0; hh < L::kHalves; ++hh) {
            tma_load_4d(stage + hh * L::kHalf, map, &full[st], 64 * hh, g, kBlk * ja, b);
            tma_load_4d(stage + hh * L::kHalf + L::kHalf / 2, map, &full[st], 64 * hh, g, kBlk * jb, b);
          }
        }
      } else {
        const int ct = t - n_blk_t;
        const int grp = ct < nct0 ? 0 : 1;
        const int cb = (grp == 0 ? ct : ct - nct0) * kKeys;
        const int mg = grp == 0 ? m0 : m1;
        const int ncol = min(kKeys, (grp == 0 ? c0 : c1) - cb);
        const int32_t *cl = a.col_idx + (grp == 0 ? lr0 : lr1) * static_cast<size_t>(a.max_col);
        const int last_row = min(kBlk * mg + kBlk - 1, a.S - 1);
        int pos[kKeys / 32];
#pragma unroll
        for (int i = 0; i < kKeys / 32; ++i) {
          const int x = lane + 32 * i;
          int j = x < ncol ? cl[cb + x] : -1;
          DSA_CHECK(x >= ncol || (j >= 0 && j < a.S));
          if (j < 0 || j > last_row) j = -1;
          pos[i] = j;
        }
        if (is_k) {
          TileMeta *md = &meta[t % kMetaRing];
          bool below = true;   // no key after the first row of block mg: no causal masking
#pragma unroll
          for (int i = 0; i < kKeys / 32; ++i) {
            md->pos[lane + 32 * i] = pos[i];
            const uint32_t ne = __ballot_sync(kFull, pos[i] >= 0);
            if (lane == 0) md->nonempty[i] = ne;
            below = below && pos[i] <= kBlk * mg;
          }
          below = __all_sync(kFull, below);
          if (lane == 0) {
            md->kind = 1;
            md->mask = HP ? 0xF : (grp == 0 ? 0x3 : 0xC);
            md->blk[0] = md->blk[1] = -1;
            md->below = below ? 1 : 0;
          }
        }
        // Eight lanes per key row, one 16-byte chunk cc of a 64-dim half each, so one
        // instruction of the warp copies four whole 128-byte row segments (rows 4r ..
        // 4r + 3; row x's position is held by lane x % 32 in pos[x / 32]); chunk cc of
        // row x lands at chunk cc ^ (x & 7) of its swizzled 128-byte row.
        const int sub = lane >> 3, cc = lane & 7;
#pragma unroll
        for (int r = 0; r < kKeys / 4; ++r) {
          const int x = 4 * r + sub;
          const int j = __shfl_sync(kFull, pos[r >> 3], x & 31);
          const uint16_t *row = src + static_cast<size_t>(j) * krow + cc * 8;
#pragma unroll
          for (int hh = 0; hh < L::kHalves; ++hh) {
            unsigned char *dst = stage + hh * L::kHalf + x * 128 + ((cc ^ (x & 7)) << 4);
            if (j >= 0) cp_async_16(dst, row + 64 * hh);
            else *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
          }
        }
        // the stage completes once every lane's copies have landed; the producer goes on
        // to the next tile meanwhile (the consumer orders them for the tensor core)
        fence_proxy_async_smem();   // the zero fills
        cp_async_mbar_arrive(&full[st]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[st]);
      }
      ++issued;
    }
    if (*abort_flag && lane == 0) {
      // let this CTA's bulk copies land before it exits
      for (int t = max(0, issued - NS); t < issued; ++t)
        drain_wait(&full[t % NS], (t / NS) & 1, 200000000ull);
      if (is_k) drain_wait(q_full, 0, 200000000ull);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16_f32(kRowsQ, kKeys, false, false);
      constexpr uint32_t id_pv = idesc_bf16_f32(kRowsQ, D, false, true);
      const uint32_t sQ = smem_u32(sm + L::oQ);
      const uint32_t sK = smem_u32(sm + L::oK);
      const uint32_t sV = smem_u32(sm + L::oV);
      auto issue_qk = [&](int t) -> bool {
        const int st = t % kKS;
        if (!tc_wait(&k_full[st], (t / kKS) & 1, wc)) return false;
        tc_fence_after();
        fence_proxy_async_smem();   // gathered rows were written by cp.async (generic proxy)
        const uint32_t d = tmem + static_cast<uint32_t>((t % kSB) * kKeys);
        const uint32_t kbase = sK + st * L::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(sQ + (kk >> 2) * L::kQHalf + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(kbase + (kk >> 2) * L::kHalf + (kk & 3) * 32, 16, 1024);
          tc_mma(d, ad, bd, id_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[t % kSB]);
        tc_commit(&k_empty[st]);
        return true;
      };
      auto issue_pv = [&](int t) -> bool {
        const int st = t % kVS;
        if (!tc_wait(&v_full[st], (t / kVS) & 1, wc)) return false;
        tc_fence_after();
        fence_proxy_async_smem();
        const uint32_t vbase = sV + st * L::kTile;
        const uint32_t pcol = tmem + static_cast<uint32_t>((t % kSB) * kKeys);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint64_t bd = sdesc_sw128(vbase + kk * 2048, L::kHalf, 1024);
          tc_mma_ts(tmem + L::cO, pcol + kk * 8, bd, id_pv, (t > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&pv_done[t % kSB]);
        tc_commit(&v_empty[st]);
        return true;
      };
      // Q K^T runs kSB tiles ahead; Q K^T of tile t + kSB reuses S_b right behind P V of t
      bool ok = tc_wait(q_full, 0, wc);
      for (int t = 0; ok && t < min(T, kSB); ++t) ok = issue_qk(t);
      for (int t = 0; ok && t < T; ++t) {
        if (!(ok = tc_wait(&p_full[t % kSB], (t / kSB) & 1, wc))) break;
        tc_fence_after();
        if (!(ok = issue_pv(t))) break;
        if (t + kSB < T) ok = issue_qk(t + kSB);
      }
      tc_commit(fin);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // Software-pipelined over tiles: the scores of tile t + 1 stream in from TMEM into the
    // registers that the exponentials of tile t have just consumed (half a slice at a
    // time), and their slice maximum is published right after P of tile t is released.
    const int sw = warp - 3;
    const int quarter = warp & 3;      // TMEM lanes this warp may access
    const int cs = sw >> 2;            // key slice of each tile
    const int row = quarter * 32 + lane;
    const int grp = row >> 6;
    const int qpos = kBlk * (grp == 0 ? m0 : m1) + (row & (kBlk - 1));
    const int hrow = grp == 0 ? hq0 : hq1;   // the row's query head
    const bool row_ok = qpos < a.S;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    constexpr int kOS = D / kSlices;   // O columns this warp rescales and stores
    const uint32_t o_col = tl + L::cO + static_cast<uint32_t>(cs * kOS);
    float *red = reinterpret_cast<float *>(sm + L::oRed);   // [3][kSlices][128 rows]
    uint64_t *qbar = xbar + 3 * quarter;   // this quarter's exchange barriers
    const float sl2 = a.sl2;
    const float2 sl2x2 = make_float2(sl2, sl2);
    const int last_key = min(qpos, a.S - 1);   // causal and in-sequence bound of the row
    float m_cur = -INFINITY, l = 0.f;   // softmax reference (base-2 units), this slice's row sum
    float m_o = -INFINITY;              // max that O is currently relative to
    bool ok = true;
    uint32_t sc[kSW];                   // this slice's scores (then those of the next tile)
    bool slice_dead = false;            // no key of the last published tile's slice is in
                                        // any row of this warp (warp-uniform)

    // TMEM column of 32-column part i of this slice in score buffer t % 3
    auto s_addr = [&](int t, int i) {
      return tl + static_cast<uint32_t>((t % kSB) * kKeys + kSW * cs + 32 * i);
    };
    // mask the scores of tile t once loaded, publish this slice's maximum
    auto publish_max = [&](int t) {
      const TileMeta *md = &meta[t % kMetaRing];
      const int kind = md->kind;
      const int hmask = row_ok ? (md->mask >> (2 * grp)) & 3 : 0;   // halves this row uses
      int lim = 0;
      bool below = false;
      if (kind == 0) {
        // slice cs is 64-key half cs, whose slot c holds key 64 * blk[cs] + c
        static_assert(kSW == kBlk, "one softmax slice per 64-key half");
        const bool member = (hmask >> cs) & 1;
        lim = member ? last_key - kBlk * md->blk[cs] : -1;   // slots <= lim are keys
      } else {
        below = md->below != 0;
      }
      tmem_wait_ld();
      const bool trim = kind != 0 || lim < kSW - 1;
      bool dead = false;
      if (__any_sync(kFull, trim)) {
        uint32_t valid[kSW / 32];   // bit c: slot c of 32-slot part i is a key of the row
#pragma unroll
        for (int i = 0; i < kSW / 32; ++i) {
          if (kind == 0) {
            const int li = lim - 32 * i;
            valid[i] = li < 0 ? 0u : (li >= 31 ? 0xffffffffu : (2u << li) - 1u);
          } else if (hmask == 0) {
            valid[i] = 0u;   // the tile belongs to the other query block
          } else if (below) {
            valid[i] = md->nonempty[(kSW * cs) / 32 + i];
          } else {
            uint32_t v = 0u;
            const int4 *pp = reinterpret_cast<const int4 *>(md->pos + kSW * cs + 32 * i);
#pragma unroll 1
            for (int c4 = 0; c4 < 8; ++c4) {
              const int4 j = pp[c4];
              v |= (static_cast<uint32_t>(j.x >= 0 && j.x <= qpos) << (4 * c4)) |
                   (static_cast<uint32_t>(j.y >= 0 && j.y <= qpos) << (4 * c4 + 1)) |
                   (static_cast<uint32_t>(j.z >= 0 && j.z <= qpos) << (4 * c4 + 2)) |
                   (static_cast<uint32_t>(j.w >= 0 && j.w <= qpos) << (4 * c4 + 3));
            }
            valid[i] = v;
          }
        }
        uint32_t any = 0u;
#pragma unroll
        for (int i = 0; i < kSW / 32; ++i) any |= valid[i];
        // a slice no row of the warp uses (the other query block's column tile, or a
        // 64-key block only the other block lists) needs neither masking nor exponentials
        dead = __all_sync(kFull, any == 0u);
        if (!dead) {
#pragma unroll
          for (int i = 0; i < kSW / 32; ++i) {
            if (__any_sync(kFull, valid[i] != 0xffffffffu)) {
#pragma unroll
              for (int c = 0; c < 32; ++c)
                sc[32 * i + c] = (valid[i] >> c) & 1u ? sc[32 * i + c] : __float_as_uint(-INFINITY);
            }
          }
        }
      }
      float m = -INFINITY;
      if (!dead) {
        float mx[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) mx[i] = -INFINITY;
#pragma unroll
        for (int c = 0; c < kSW; c += 2)
          mx[(c >> 1) & 3] = fmax3(mx[(c >> 1) & 3], __uint_as_float(sc[c]), __uint_as_float(sc[c + 1]));
        m = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
      }
      slice_dead = dead;
      red[((t & 1) * kSlices + cs) * kRowsQ + row] = m;
      __syncwarp();
      if (lane == 0) mbar_arrive(&qbar[t & 1]);
    };
    // tile t: row max from the row's slices, P, row sum, prefetch of tile t + 1's scores,
    // rescale, release of P
    auto finish_tile = [&](int t) -> bool {
      const bool more = t + 1 < T;
      const bool dead = slice_dead;   // publish_max(t + 1) below overwrites it
      // tile t's phase on its exchange barrier is its (t / 2)-th; the warp itself waited
      // the one before, and the one after needs this warp's own arrival
      if (!warp_wait(&qbar[t & 1], (t >> 1) & 1, wc)) return false;
      const float *rr = red + (t & 1) * kSlices * kRowsQ + row;
      float mraw = rr[0];
#pragma unroll
      for (int i = 1; i < kSlices; ++i) mraw = fmaxf(mraw, rr[i * kRowsQ]);
      const float mt = mraw * sl2;
      // sl2 > 0: same order as the scaled scores; -inf + slack stays -inf
      if (mt > m_cur + kRescaleSlack) {
        if (m_cur != -INFINITY) l *= fast_exp2(m_cur - mt);
        m_cur = mt;
      }
      // probabilities -> kSW / 2 bf16 pairs at columns (kSW / 2) cs.. of S_b, the first
      // half of the tile's score columns; every slice of the tile was loaded before its
      // maximum was published
      const float nm = m_cur == -INFINITY ? 0.f : -m_cur;   // no key yet: every s is -inf
      const float2 nm2 = make_float2(nm, nm);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
      const uint32_t pcol = tl + static_cast<uint32_t>((t % kSB) * kKeys + (kSW / 2) * cs);
      bool got = true;
#pragma unroll
      for (int i = 0; i < kSW / 32; ++i) {
        uint32_t pk[16];
        if (dead) {   // every probability of the slice is 0
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[c] = 0u;
        } else {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const int k = 32 * i + c;
            const float2 y = ffma2(make_float2(__uint_as_float(sc[k]), __uint_as_float(sc[k + 1])), sl2x2, nm2);
            const float2 e = make_float2(fast_exp2(y.x), fast_exp2(y.y));
            if ((c >> 1) & 1) acc1 = fadd2(acc1, e);
            else acc0 = fadd2(acc0, e);
            pk[c >> 1] = pack_bf16x2(e.x, e.y);
          }
        }
        tmem_st16(pcol + 16 * i, pk);
        if (more) {   // part i of this slice is free: bring in tile t + 1's
          if (i == 0) {
            got = warp_wait(&s_full[(t + 1) % kSB], ((t + 1) / kSB) & 1, wc);
            if (got) tc_fence_after();
          }
          if (got) tmem_ld32(s_addr(t + 1, i), sc + 32 * i);
        }
      }
      const float2 as = fadd2(acc0, acc1);
      l += as.x + as.y;
      // O to the current max, once P V of the previous tile has retired.  P V of tile k
      // completes phase k / 3 of pv_done[k % 3]; P V of tile t - 4 has retired (Q K^T of
      // tile t came after it), so the parity names the phase of tile t - 1 exactly.
      const bool stale = m_o != -INFINITY && m_o < m_cur;
      if (__any_sync(kFull, stale)) {
        const int tp = t - 1;   // >= 0: O has a max only after a tile
        if (!warp_wait(&pv_done[tp % kSB], (tp / kSB) & 1, wc)) return false;
        tc_fence_after();
        const float f = stale ? fast_exp2(m_o - m_cur) : 1.f;
        const float2 f2 = make_float2(f, f);
#pragma unroll 1
        for (int c16 = 0; c16 < kOS; c16 += 16) {
          uint32_t o[16];
          tmem_ld16(o_col + c16, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            const float2 y = fmul2(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), f2);
            o[i] = __float_as_uint(y.x);
            o[i + 1] = __float_as_uint(y.y);
          }
          tmem_st16(o_col + c16, o);
        }
      }
      m_o = m_cur;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t % kSB]);
      if (!got) return false;
      if (more) publish_max(t + 1);
      return true;
    };
    if (T > 0) {
      if (warp_wait(&s_full[0], 0, wc)) {
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < kSW / 32; ++i) tmem_ld32(s_addr(0, i), sc + 32 * i);
        publish_max(0);
      } else {
        ok = false;
      }
    }
    for (int t = 0; ok && t < T; ++t) ok = finish_tile(t);
    // epilogue: the last P V, then the row sums of the row's slices
    const bool have_o = ok && T > 0 && warp_wait(&pv_done[(T - 1) % kSB], ((T - 1) / kSB) & 1, wc);
    red[(2 * kSlices + cs) * kRowsQ + row] = l;
    __syncwarp();
    if (lane == 0) mbar_arrive(&qbar[2]);
    const bool have_l = warp_wait(&qbar[2], 0, wc);
    const float *rr = red + 2 * kSlices * kRowsQ + row;
    float lt = rr[0];
#pragma unroll
    for (int i = 1; i < kSlices; ++i) lt += rr[i * kRowsQ];
    // warp-uniform: the TMEM load is collective.  A CTA that gave up stores zeros.
    const bool ld_ok = have_o && have_l && !*abort_flag;
    const bool good = ld_ok && lt > 0.f;
    const float inv = good ? 1.f / lt : 0.f;
    uint32_t o[kOS];
    if (ld_ok) {
      tc_fence_after();
#pragma unroll
      for (int i = 0; i < kOS / 32; ++i) tmem_ld32(o_col + 32 * i, o + 32 * i);
      tmem_wait_ld();
    }
    if (row_ok) {
      uint32_t w[kOS / 2];
#pragma unroll
      for (int i = 0; i < kOS / 2; ++i)
        w[i] = good ? pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv) : 0u;
      uint4 *dst = reinterpret_cast<uint4 *>(a.out + ((static_cast<size_t>(b) * a.S + qpos) * a.H_q + hrow) * D +
                                             cs * kOS);
#pragma unroll
      for (int i = 0; i < kOS / 8; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      if (cs == 0 && a.lse)
        a.lse[(static_cast<size_t>(b) * a.H_q + hrow) * a.S + qpos] = good ? (m_cur + log2f(lt)) * kLn2 : -INFINITY;
    }
  }

}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcArgs a) {
  using L = Layout<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::oBar);
  uint64_t *k_full = bars, *k_empty = k_full + kKS;
  uint64_t *v_full = k_empty + kKS, *v_empty = v_full + kVS;
  uint64_t *s_full = v_empty + kVS, *p_full = s_full + kSB;
  uint64_t *pv_done = p_full + kSB, *q_full = pv_done + kSB, *fin = q_full + 1;
  uint64_t *xbar = fin + 1;   // [4 quarters][3]: row-max exchange by tile parity, row sums
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::oMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::oMisc + 4);
  int *n_blk_tiles_s = reinterpret_cast<int *>(sm + L::oMisc + 8);
  uint32_t *bm0 = reinterpret_cast<uint32_t *>(sm + L::oBits);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // longest rows first; the G query heads of one KV head side by side, so the CTAs that
  // read the same key and value rows (for lists shared by the heads, the same rows)
  // run together and share them through L2
  const int n_pairs = (a.n_qblk + 1) / 2;
  const int G = a.H_q / a.H_kv;
  const int hl = static_cast<int>(blockIdx.x) % G;   // query head within the KV head
  const int p = n_pairs - 1 - static_cast<int>(blockIdx.x) / G;
  const int g = blockIdx.y, b = blockIdx.z;
  // The CTA's 128 rows are two 64-row groups, each one (query head, query block).  The
  // two CTAs of query heads hA = 2i, hA + 1 of a KV head at pair p share the four rows
  // (hA, hA + 1) x (2p, 2p + 1): when both heads list the same blocks and columns for
  // both query blocks (lists made once for every head, as the InfiniteHiP ones are), CTA
  // hl & 1 takes query block 2p + (hl & 1) of both heads, so that every tile serves all
  // 128 rows; otherwise each takes its own head's blocks 2p and 2p + 1.
  const int hA = g * G + (hl & ~1);
  const bool quad = (hl | 1) < G && 2 * p + 1 < a.n_qblk;
  bool differ = !quad;
  if (quad) {
    const size_t rA = (static_cast<size_t>(b) * a.H_q + hA) * a.n_qblk, rB = rA + a.n_qblk;
#pragma unroll 1
    for (int m = 2 * p; m <= 2 * p + 1 && !differ; ++m) {
      const int nb = min(max(a.blk_cnt[rA + m], 0), a.max_blk), nc = min(max(a.col_cnt[rA + m], 0), a.max_col);
      if (nb != min(max(a.blk_cnt[rB + m], 0), a.max_blk) || nc != min(max(a.col_cnt[rB + m], 0), a.max_col)) {
        differ = true;
        break;
      }
      const int32_t *ba = a.blk_idx + (rA + m) * static_cast<size_t>(a.max_blk);
      const int32_t *bb = a.blk_idx + (rB + m) * static_cast<size_t>(a.max_blk);
      for (int i = tid; i < nb; i += kThreads) differ |= ba[i] != bb[i];
      if (nc > 0) {
        const int32_t *ca = a.col_idx + (rA + m) * static_cast<size_t>(a.max_col);
        const int32_t *cb = a.col_idx + (rB + m) * static_cast<size_t>(a.max_col);
        for (int i = tid; i < nc; i += kThreads) differ |= ca[i] != cb[i];
      }
    }
  }

  if (tid == 0) {
    for (int i = 0; i < 2 * kKS + 2 * kVS; ++i) mbar_init(&bars[i], 1);
    for (int i = 0; i < kSB; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kSmWarps);   // one arrival per softmax warp
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(fin, 1);
    for (int i = 0; i < 4 * 3; ++i) mbar_init(&xbar[i], kSlices);   // one arrival per key slice
    *abort_flag = 0;
    *n_blk_tiles_s = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  for (int w = tid; w < 2 * a.n_words; w += kThreads) bm0[w] = 0u;
  const bool head_pair = __syncthreads_or(differ ? 1 : 0) == 0;
  if (head_pair) tc_cta<D, true>(a, sm, p, g, b, hl, hA);
  else tc_cta<D, false>(a, sm, p, g, b, hl, hA);
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    if (lane == 0) drain_wait(fin, 0, 1000000000ull);   // every MMA retired before TMEM is freed
    __syncwarp();
    tmem_dealloc(*tmem_slot, kTmemCols);
  }
  if (tid == 0 && *abort_flag) atomicExch(&g_prefill_tc_error, 1);
}

}  // namespace

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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
bool make_bshd_map(CUtensorMap *m, const void *base, int D, int H, int S, int B, int rows) {
  auto enc = tensor_map_encoder();
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

namespace {

template <int D>
cudaError_t launch_tc_d(const PrefillArgs &pa, cudaStream_t s) {
  TcArgs a;
  std::memset(&a, 0, sizeof(a));
  if (!make_bshd_map(&a.tq, pa.q, D, pa.H_q, pa.S, pa.B, kBlk) ||
      !make_bshd_map(&a.tk, pa.k, D, pa.H_kv, pa.S, pa.B, kBlk) ||
      !make_bshd_map(&a.tv, pa.v, D, pa.H_kv, pa.S, pa.B, kBlk))
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
  a.n_qblk = (pa.S + kBlk - 1) / kBlk;
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
  dim3 grid((a.n_qblk + 1) / 2 * (pa.H_q / pa.H_kv), pa.H_kv, pa.B);
  {
    ProfScope ps("prefill_attention_tc", s);
    kern<<<grid, kThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

// The kernel orders scores by their raw value, which needs a positive scale; it also
// needs D in {64, 128}, the bitmaps of one query-block pair in shared memory and the
// driver's tensor-map encoder.
int prefill_tc_check(const PrefillArgs &a) {
  if (a.D != 64 && a.D != 128) return fail(DSA_ERR_UNSUPPORTED, "D=%d not in {64, 128}", a.D);
  if (!(a.scale > 0.f)) return fail(DSA_ERR_INVALID_ARG, "scale=%g must be positive", a.scale);
  const int n_qblk = (a.S + kBlk - 1) / kBlk;
  const size_t smem = a.D == 128 ? Layout<128>::bytes((n_qblk + 31) / 32)
                                 : Layout<64>::bytes((n_qblk + 31) / 32);
  if (smem > 227 * 1024)
    return fail(DSA_ERR_UNSUPPORTED, "S=%d: %zu bytes of shared memory per CTA > 227 KiB", a.S, smem);
  if (tensor_map_encoder() == nullptr)
    return fail(DSA_ERR_UNSUPPORTED, "the driver offers no cuTensorMapEncodeTiled entry point");
  return DSA_OK;
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
  const int w = vs_tc_device_error();   // the vertical-slash estimate's word
  if (w < 0) return fail(DSA_ERR_CUDA, "reading the estimate's device error word");
  // checked builds: out-of-range device-side inputs met by the kernels
  int chk = 0;
  const int words[5] = {decode_check_word(), decode_mma_check_word(), hip_select_check_word(),
                        stage_tc_check_word(), prefill_tc_check_word()};
  for (int x : words) {
    if (x < 0) return fail(DSA_ERR_CUDA, "reading a device check word");
    chk |= x;
  }
  *code = v | (w << 1) | (chk ? 4 : 0);
  if (chk)
    return fail(DSA_ERR_DEVICE_CHECK, "a kernel met a device-side input outside its range "
                                      "(length, count, selected position or list entry)");
  return DSA_OK;
}

namespace dsa {
int prefill_tc_set_wait_limit(unsigned long long ns) {
  return cudaMemcpyToSymbol(g_wait_limit_ns, &ns, sizeof(ns)) == cudaSuccess ? 0 : -1;
}
}  // namespace dsa

extern "C" int dsa_set_wait_limit(unsigned long long ns) {
  using namespace dsa;
  clear_error();
  const unsigned long long v = ns ? ns : kWaitLimitNs;
  if (prefill_tc_set_wait_limit(v) || vs_tc_set_wait_limit(v))
    return fail(DSA_ERR_CUDA, "setting the wait limit of the tensor-core kernels");
  return DSA_OK;
}
