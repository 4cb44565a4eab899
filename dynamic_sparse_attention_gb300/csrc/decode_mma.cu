// Sparse GQA decode on warp-level tensor cores, one thread-block cluster per
// (batch row b, KV head g).
//
// Source: "InfiniteHiP: Extending Language Model Context Up to 3 Million Tokens on a
// Single GPU" (paper-graph-ui summary), section 3.4 "Block Sparse Attention
// Implementation" (decoding: split the keys across thread blocks, partial softmax,
// final reduction) and "Formal Background" (softmax attention).
//
// Decode is bound by the latency of gathering a few thousand scattered K/V rows, not
// by arithmetic.  The design therefore puts every gather in flight early and keeps
// the per-key work on tensor cores:
//  * the cluster's CTAs (up to 16) split the attended keys of (b, g) in two parts: the
//    sink and window keys, whose positions follow from kv_len alone, and the selected
//    slots of sel_idx.  The selection's last kernel lets this grid start as soon as it
//    starts itself, so a CTA gathers and scores its sink / window keys while the
//    selection finishes, and only then waits for sel_idx (griddepcontrol.wait) and
//    gathers its selected keys.  Inside a CTA each warp owns every NW-th 16-key
//    sub-tile, gathers it (16-byte cp.async, a token's row for head g is 2*D contiguous
//    bytes) into its own shared-memory ring and keeps its own online softmax; rows of
//    sub-tiles past the ring's first fill are requested from L2 in the round of that
//    fill.  Eight warps with two slots each hold a 1M-context CTA's selected sub-tiles
//    in one round, but at about 100 registers a thread only two such CTAs share an SM,
//    so they are launched only when every cluster of the launch fits the GPU at once;
//    otherwise four warps with up to four slots;
//  * S = Q K^T and O += P V are mma.sync m16n8k16 (bf16 in, fp32 accumulate): the
//    G*T_q query rows (at most 16) of the KV head are the M = 16 rows, keys and head
//    dimensions the N and K sides; P goes from the S accumulators straight into the A
//    operand of the P V product;
//  * the running max is exact (the row's largest probability is exactly 1) and the
//    row sum adds the same bf16-rounded probabilities that enter P V;
//  * at the end the warps of a CTA merge in shared memory (over the drained rings) and
//    the CTAs of the cluster merge through distributed shared memory (log-sum-exp
//    weights; a few threads per output read all CTAs' partials in one round);
//    nothing goes through HBM but the K/V rows, the query and the output.
//  * FP8 E4M3 keys and values (a bf16 query, D = 128; the "FP8 KV cache data type" of
//    the InfiniteHiP summary's throughput runs): a sub-tile is 4 KiB, so up to six are
//    in flight per warp -- every sub-tile of a 1M-context range at once -- and the
//    products run as fp16 mma.sync (E4M3 and bf16 values are fp16 values; P rounds to
//    fp16).  The bytes go from shared memory straight into fragments: Q K^T takes each
//    16-dim k-step in the order (4t, 4t+1 | 4t+2, 4t+3) for fragment columns
//    (2t, 2t+1 | 2t+8, 2t+9), so one 32-bit load of four codes is a whole B fragment,
//    and the sub-tile's key order is permuted the same way (n-tile i, column 2t + e is
//    key 4t + 2i + e), so the P V fragment of a head dimension is four codes of
//    consecutive keys.
#include <algorithm>

#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "mma_sync.cuh"
#include "profile.h"

namespace dsa {

DSA_CHECK_WORD(decode_mma_check_word)

namespace {

// Ring slots: a bf16 sub-tile (K and V rows of 16 keys) is 8 KiB at d = 128, an FP8 one
// 4 KiB.  (Eight warps for FP8 rows measured slower: the registers then spill.)
constexpr int kST = 16;      // keys per warp sub-tile
constexpr int kMaxBuf = 4;   // sub-tiles in flight per warp, at most (bf16 rows, four warps)
constexpr int kMaxBuf8W = 2; // the same with eight warps
constexpr int kMaxBuf8 = 6;  // the same for FP8 rows
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Shared rows are D bf16 with the 16-byte pieces of key row k stored at piece index
// c ^ (k & 7): the eight rows an ldmatrix reads at one piece index hit eight
// different bank groups.  The warp and CTA partials reuse the rings once every gather
// has landed.
template <int D, bool FP8, int NW>
struct MmaSmem {
  static constexpr int kWarps = NW;
  static constexpr int kRowBytes = FP8 ? D : 2 * D;      // one key row of one head
  static constexpr int kSlotBytes = 2 * kST * kRowBytes;   // K rows then V rows of one sub-tile
  __host__ __device__ static size_t ring_bytes(int nbuf) {
    return static_cast<size_t>(kWarps) * nbuf * kSlotBytes;
  }
  __host__ __device__ static size_t part_bytes(int R) {             // warp partials, CTA partial, merge weights
    return (static_cast<size_t>(kWarps + 1) * R * (D + 2) + static_cast<size_t>(kWarps) * R) * 4;
  }
  __host__ __device__ static size_t rings_or_parts(int nbuf, int R) {
    return ring_bytes(nbuf) > part_bytes(R) ? ring_bytes(nbuf) : part_bytes(R);
  }
  static size_t bytes(int kps, int R, int nbuf) {
    return rings_or_parts(nbuf, R) + static_cast<size_t>(kps) * 4;   // + key positions
  }
};

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(smem_dst)),
               "l"(gmem_src));
}

// element offset of piece c (8 bf16) of key row k in a swizzled tile
template <int D>
__device__ __forceinline__ int sw_off(int k, int c) {
  return k * D + ((c ^ (k & 7)) << 3);
}

__device__ __forceinline__ float bf16r(float x) {   // x rounded to bf16 (nearest even)
  return __uint_as_float(static_cast<uint32_t>(f32_to_bf16(x)) << 16);
}

__device__ __forceinline__ float f16r(float x) {    // x rounded to fp16 (nearest even)
  return __half2float(__float2half_rn(x));
}

// byte offset of 16-byte piece c of key row k in a swizzled FP8 tile (128-byte rows)
__device__ __forceinline__ int sw8_off(int k, int c) { return k * 128 + ((c ^ (k & 7)) << 4); }

template <int D, int NBUF, bool FP8, int NW>
__global__ void __launch_bounds__(NW * 32) decode_mma_kernel(DecodeArgs a) {
  namespace cg = cooperative_groups;
  using SM = MmaSmem<D, FP8, NW>;
  constexpr int kWarps = SM::kWarps;
  constexpr int kThreads = kWarps * 32;
  static_assert(!FP8 || D == 128, "FP8 rows: D = 128");
  constexpr int KS = D / 16;   // k-steps of Q K^T
  constexpr int NT = D / 8;    // n-tiles of P V
  constexpr int CH = SM::kRowBytes / 16;   // 16-byte pieces per K or V row
  extern __shared__ __align__(16) unsigned char smem[];
  const int G = a.H_q / a.H_kv;
  const int R = G * a.T_q;     // <= 16
  unsigned char *ring = smem;
  float *s_part = reinterpret_cast<float *>(smem);   // over the drained rings
  int *s_pos = reinterpret_cast<int *>(smem + SM::rings_or_parts(NBUF, R));

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int C = static_cast<int>(cluster.num_blocks());
  const int g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;
  uint32_t qa[KS][4];   // the query rows as A fragments (loaded below)
  // Keys of this CTA: fixed keys (sink and window, whose positions follow from kv_len
  // alone) [rank * fix_per, +fix_per) of the virtual order sink | window, and selected
  // slots [rank * sel_per, +sel_per).  The fixed keys are gathered and scored before
  // the wait on the previous kernel (the selection's last kernel, which writes
  // sel_idx / sel_cnt and lets this grid start early); only the selected ones after it.
  const int kv_raw = a.kv_len[b];
  DSA_CHECK(kv_raw >= 0 && kv_raw <= a.T_max);
  const int Tb = min(max(kv_raw, 0), a.T_max);
  const int n_s = min(a.n_sink, Tb);
  const int w0 = max(a.n_sink, Tb - a.n_stream);
  const int n_w = max(0, Tb - w0);
  const int f_begin = rank * a.fix_per;
  const int f_end = min(n_s + n_w, f_begin + a.fix_per);
  const int nf_sub = f_end > f_begin ? (f_end - f_begin + kST - 1) / kST : 0;
  int *s_posf = s_pos;                 // [fix_per]
  int *s_poss = s_pos + a.fix_per;     // [sel_per]
  for (int i = tid; i < a.fix_per; i += kThreads) {
    const int f = f_begin + i;
    int pos = -1;
    if (f < f_end) pos = f < n_s ? f : w0 + (f - n_s);
    s_posf[i] = (pos >= 0 && pos < Tb) ? pos : -1;
  }
  __syncthreads();
  constexpr int kEl = FP8 ? 1 : 2;   // bytes per K / V element
  const unsigned char *kbase = static_cast<const unsigned char *>(a.k) +
                               (static_cast<size_t>(b) * a.T_max * a.H_kv * D + static_cast<size_t>(g) * D) * kEl;
  const unsigned char *vbase = static_cast<const unsigned char *>(a.v) +
                               (static_cast<size_t>(b) * a.T_max * a.H_kv * D + static_cast<size_t>(g) * D) * kEl;
  const size_t row_stride = static_cast<size_t>(a.H_kv) * D * kEl;   // bytes
  const float sl2 = a.scale * kLog2e;

  unsigned char *wring = ring + warp * NBUF * SM::kSlotBytes;
  // sub-tile j (positions pj[j * kST ...], n_sub of them) -> ring slot `slot`; one commit
  // group per call
  auto issue = [&](const int *pos_arr, int j, int n_sub, int slot) {
    if (j < n_sub) {
      unsigned char *sk = wring + slot * SM::kSlotBytes;
      unsigned char *sv = sk + kST * SM::kRowBytes;
      const int *pj = pos_arr + j * kST;
#pragma unroll
      for (int e = lane; e < kST * CH; e += 32) {
        const int key = e / CH, c = e - key * CH;
        const int pos = pj[key];
        const int off = FP8 ? sw8_off(key, c) : 2 * sw_off<D>(key, c);
        unsigned char *dk = sk + off;
        unsigned char *dv = sv + off;
        if (pos >= 0) {
          cp_async16(dk, kbase + static_cast<size_t>(pos) * row_stride + c * 16);
          cp_async16(dv, vbase + static_cast<size_t>(pos) * row_stride + c * 16);
        } else {
          *reinterpret_cast<uint4 *>(dk) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4 *>(dv) = make_uint4(0, 0, 0, 0);
        }
      }
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };

  float o[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows gq and gq + 8

  // one landed sub-tile into the running softmax of this warp
  auto consume = [&](const int *pj, int slot) {
    const unsigned char *sk = wring + slot * SM::kSlotBytes;
    const unsigned char *sv = sk + kST * SM::kRowBytes;
    // S = Q K^T: two n-tiles of 8 keys
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if constexpr (FP8) {
      // n-tile i, column gq holds key 4 (gq >> 1) + (gq & 1) + 2i; one 32-bit load gives
      // that key's dims (4t .. 4t+3) of k-step ks: b0 = the first two, b1 = the last two
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int key = 4 * (gq >> 1) + (gq & 1) + 2 * nt;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint32_t w = *reinterpret_cast<const uint32_t *>(sk + sw8_off(key, ks) + 4 * tq);
          mma_16816_f16(s[nt], qa[ks], e4m3x2_to_f16x2(w), e4m3x2_to_f16x2(w >> 16));
        }
      }
    } else {
      const int mtx = lane >> 3, rr = lane & 7;
      const int key = (mtx >> 1) * 8 + rr;
      const uint16_t *sk16 = reinterpret_cast<const uint16_t *>(sk);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t bk[4];
        ldsm_x4(bk, sk16 + sw_off<D>(key, 2 * ks + (mtx & 1)));
        mma_16816(s[0], qa[ks], bk[0], bk[1]);
        mma_16816(s[1], qa[ks], bk[2], bk[3]);
      }
    }
    // scale, mask keys without a position, exact running max per row
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = FP8 ? 4 * tq + 2 * nt + (e & 1) : nt * 8 + 2 * tq + (e & 1);
        const float v = pj[key] >= 0 ? s[nt][e] * sl2 : -INFINITY;
        s[nt][e] = v;
        if (e < 2) mx0 = fmaxf(mx0, v);
        else mx1 = fmaxf(mx1, v);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    const float al0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - n0);
    const float al1 = (m1 == -INFINITY) ? 0.f : exp2f(m1 - n1);
    m0 = n0;
    m1 = n1;
    // probabilities, rounded once to the operand type (bf16, or fp16 with FP8 rows): the
    // same values feed P V and the row sums
    auto rnd = [](float x) { return FP8 ? f16r(x) : bf16r(x); };
    auto pack = [](float lo, float hi) { return FP8 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi); };
    uint32_t pa[4];
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const float p0 = n0 == -INFINITY ? 0.f : rnd(exp2f(s[nt][0] - n0));
      const float p1 = n0 == -INFINITY ? 0.f : rnd(exp2f(s[nt][1] - n0));
      const float p2 = n1 == -INFINITY ? 0.f : rnd(exp2f(s[nt][2] - n1));
      const float p3 = n1 == -INFINITY ? 0.f : rnd(exp2f(s[nt][3] - n1));
      ps0 += p0 + p1;
      ps1 += p2 + p3;
      pa[2 * nt] = pack(p0, p1);       // a0 (n-tile 0) / a2 (n-tile 1): row gq
      pa[2 * nt + 1] = pack(p2, p3);   // a1 / a3: row gq + 8
    }
    ps0 += __shfl_xor_sync(kFull, ps0, 1);
    ps0 += __shfl_xor_sync(kFull, ps0, 2);
    ps1 += __shfl_xor_sync(kFull, ps1, 1);
    ps1 += __shfl_xor_sync(kFull, ps1, 2);
    l0 = l0 * al0 + ps0;
    l1 = l1 * al1 + ps1;
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      o[i][0] *= al0;
      o[i][1] *= al0;
      o[i][2] *= al1;
      o[i][3] *= al1;
    }
    // O += P V: V rows (keys) are the K side, head dimensions the N side
    const uint32_t pfrag[4] = {pa[0], pa[1], pa[2], pa[3]};
    if constexpr (FP8) {
      // fragment rows (2t, 2t+1 | 2t+8, 2t+9) are keys 4t .. 4t+3; column gq of n-tile i is
      // head dim 8i + gq: four codes, one per key
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const int d = 8 * i + gq;
        uint32_t x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) x[u] = sv[sw8_off(4 * tq + u, d >> 4) + (d & 15)];
        mma_16816_f16(o[i], pfrag, e4m3x2_to_f16x2(x[0] | (x[1] << 8)),
                      e4m3x2_to_f16x2(x[2] | (x[3] << 8)));
      }
    } else {
      const int mtx = lane >> 3, rr = lane & 7;
      const int key = (mtx & 1) * 8 + rr;
      const uint16_t *sv16 = reinterpret_cast<const uint16_t *>(sv);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t bv[4];
        ldsm_x4_trans(bv, sv16 + sw_off<D>(key, 2 * dp + (mtx >> 1)));
        mma_16816(o[2 * dp], pfrag, bv[0], bv[1]);
        mma_16816(o[2 * dp + 1], pfrag, bv[2], bv[3]);
      }
    }
  };
  // a run of sub-tiles j = warp, warp + kWarps, ... < n_sub through this warp's ring:
  // prime() fills the ring, drain() consumes and refills it
  auto prime = [&](const int *pos_arr, int n_sub) {
#pragma unroll
    for (int s = 0; s < NBUF; ++s) issue(pos_arr, warp + s * kWarps, n_sub, s);
  };
  auto drain = [&](const int *pos_arr, int n_sub) {
    for (int it = 0, j = warp; j < n_sub; ++it, j += kWarps) {
      const int slot = it % NBUF;
      asm volatile("cp.async.wait_group %0;\n" ::"n"(NBUF - 1) : "memory");
      __syncwarp();
      consume(pos_arr + j * kST, slot);
      __syncwarp();
      issue(pos_arr, j + NBUF * kWarps, n_sub, slot);
    }
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    __syncwarp();
  };

  prime(s_posf, nf_sub);   // sink and window keys, while the selection finishes
  // the query rows as A fragments (row r = t * G + j of head g * G + j; rows >= R zero),
  // loaded while the first sink / window rows are in flight
  {
    const uint16_t *q = static_cast<const uint16_t *>(a.q);
    auto qpair = [&](int r, int d) -> uint32_t {
      if (r >= R) return 0u;
      const int t = r / G, h = g * G + (r - t * G);
      const uint32_t w = *reinterpret_cast<const uint32_t *>(
          q + ((static_cast<size_t>(b) * a.T_q + t) * a.H_q + h) * D + d);
      if constexpr (FP8) return pack_f16x2(bf16_lo(w), bf16_hi(w));   // exact but for tiny values
      else return w;
    };
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      // FP8: fragment columns (2t, 2t+1 | 2t+8, 2t+9) hold dims (4t, 4t+1 | 4t+2, 4t+3)
      const int d0 = FP8 ? ks * 16 + 4 * tq : ks * 16 + 2 * tq;
      const int d1 = FP8 ? d0 + 2 : d0 + 8;
      qa[ks][0] = qpair(gq, d0);
      qa[ks][1] = qpair(gq + 8, d0);
      qa[ks][2] = qpair(gq, d1);
      qa[ks][3] = qpair(gq + 8, d1);
    }
  }
  drain(s_posf, nf_sub);

  grid_dep_wait();
  const int32_t *sel = a.sel_idx + static_cast<size_t>(b) * a.max_sel;
  const int cnt_raw = a.sel_cnt[b];
  DSA_CHECK(cnt_raw >= 0 && cnt_raw <= a.max_sel);
  const int cnt = min(max(cnt_raw, 0), a.max_sel);
  const int s_begin = rank * a.sel_per;
  const int s_end = min(cnt, s_begin + a.sel_per);
  const int ns_sub = s_end > s_begin ? (s_end - s_begin + kST - 1) / kST : 0;
  for (int i = tid; i < a.sel_per; i += kThreads) {
    const int x = s_begin + i;
    int pos = x < s_end ? __ldg(sel + x) : -1;
    DSA_CHECK(x >= s_end || (pos >= a.n_sink && pos < max(a.n_sink, Tb - a.n_stream)));
    s_poss[i] = (pos >= 0 && pos < Tb) ? pos : -1;   // never read outside the row's context
  }
  __syncthreads();
  // Rows of the sub-tiles past the first ring fill of their warp are requested from L2
  // now, in the round of the first fill, so the later fills hit L2.
  {
    const int first_late = NBUF * kWarps;   // sub-tiles [0, first_late) go in the first fill
    const int n_late = ns_sub > first_late ? (ns_sub - first_late) * kST : 0;
    constexpr int kLines = (SM::kRowBytes + 127) / 128;   // 128-byte lines per row
    for (int u = tid; u < n_late * 2 * kLines; u += kThreads) {
      const int key = first_late * kST + u / (2 * kLines);
      const int rest = u % (2 * kLines);
      const int pos = s_poss[key];
      if (pos < 0) continue;
      const unsigned char *row = (rest < kLines ? kbase : vbase) + static_cast<size_t>(pos) * row_stride +
                                 128 * (rest % kLines);
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"(row));
    }
  }
  prime(s_poss, ns_sub);
  drain(s_poss, ns_sub);
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  __syncthreads();   // every ring drained: the partials below overwrite them

  // this warp's partial for the rows it holds: [warp][R][D + 2] = (acc, m, l)
  {
    float *wp = s_part + static_cast<size_t>(warp) * R * (D + 2);
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const int d = i * 8 + 2 * tq;
      if (gq < R) {
        wp[gq * (D + 2) + d] = o[i][0];
        wp[gq * (D + 2) + d + 1] = o[i][1];
      }
      if (gq + 8 < R) {
        wp[(gq + 8) * (D + 2) + d] = o[i][2];
        wp[(gq + 8) * (D + 2) + d + 1] = o[i][3];
      }
    }
    if (tq == 0) {
      if (gq < R) {
        wp[gq * (D + 2) + D] = m0;
        wp[gq * (D + 2) + D + 1] = l0;
      }
      if (gq + 8 < R) {
        wp[(gq + 8) * (D + 2) + D] = m1;
        wp[(gq + 8) * (D + 2) + D + 1] = l1;
      }
    }
  }
  __syncthreads();
  // the CTA's partial from its warps: per row the max and the warps' weights once, then
  // every element as a weighted sum
  float *cp = s_part + static_cast<size_t>(kWarps) * R * (D + 2);
  float *s_wgt = cp + static_cast<size_t>(R) * (D + 2);   // [kWarps][R]
  if (tid < R) {
    const int r = tid;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_part[(w * R + r) * (D + 2) + D]);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float m = s_part[(w * R + r) * (D + 2) + D];
      const float wgt = (m == -INFINITY) ? 0.f : exp2f(m - M);
      s_wgt[w * R + r] = wgt;
      L = fmaf(s_part[(w * R + r) * (D + 2) + D + 1], wgt, L);
    }
    cp[r * (D + 2) + D] = M;
    cp[r * (D + 2) + D + 1] = L;
  }
  __syncthreads();
  for (int e = tid; e < R * D; e += kThreads) {
    const int r = e / D, d = e - r * D;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) acc = fmaf(s_part[(w * R + r) * (D + 2) + d], s_wgt[w * R + r], acc);
    cp[r * (D + 2) + d] = acc;
  }
  cluster.sync();
  // merge across the cluster: the CTAs share the R*D outputs; tpe threads per output
  // (the most that leave one pass over this CTA's outputs), each reading the partials of
  // CTAs part, part + tpe, ... -- every remote load of the CTA is issued in one round
  const int E = R * D;
  const int per = (E + C - 1) / C;
  const int e_beg = rank * per, e_end = min(E, e_beg + per);
  int tpe = 16;
  while (tpe > 1 && (kThreads / tpe) < per) tpe >>= 1;
  const int cpt = (C + tpe - 1) / tpe;    // CTAs per thread (<= 16)
  const int part = tid & (tpe - 1);
  for (int base = e_beg; base < e_end; base += kThreads / tpe) {   // uniform trip count
    const int e = base + tid / tpe;
    const bool valid = e < e_end;
    const int r = valid ? e / D : 0, d = valid ? e - r * D : 0;
    const float *pr = cp + r * (D + 2);
    float mc[16], lc[16], oc[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int c = part + u * tpe;
      mc[u] = -INFINITY;
      lc[u] = oc[u] = 0.f;
      if (u < cpt && valid && c < C) {
        mc[u] = *cluster.map_shared_rank(pr + D, c);
        lc[u] = *cluster.map_shared_rank(pr + D + 1, c);
        oc[u] = *cluster.map_shared_rank(pr + d, c);
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int u = 0; u < 16; ++u) M = fmaxf(M, mc[u]);
    for (int x = 1; x < tpe; x <<= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, x));
    float Ls = 0.f, ov = 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      if (mc[u] != -INFINITY) {
        const float wgt = exp2f(mc[u] - M);
        Ls = fmaf(lc[u], wgt, Ls);
        ov = fmaf(oc[u], wgt, ov);
      }
    }
    for (int x = 1; x < tpe; x <<= 1) {
      Ls += __shfl_xor_sync(kFull, Ls, x);
      ov += __shfl_xor_sync(kFull, ov, x);
    }
    if (valid && part == 0) {
      const int t = r / G, h = g * G + (r - t * G);
      const size_t row = (static_cast<size_t>(b) * a.T_q + t) * a.H_q + h;
      static_cast<uint16_t *>(a.out)[row * D + d] = f32_to_bf16(Ls > 0.f ? ov / Ls : 0.f);
      if (a.lse && d == 0) a.lse[row] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
    }
  }
  cluster.sync();   // keep this CTA's shared memory until every reader is done
}

// Launch shape of the cluster kernel: warps per CTA, cluster size and ring cap.
struct MmaShape {
  int nw, C, cap;
};

template <int D, bool FP8, int NW>
struct MmaKernels {
  using Kern = void (*)(DecodeArgs);
  static Kern get(int nbuf) {
    if constexpr (FP8) {
      switch (nbuf) {
        case 1: return decode_mma_kernel<D, 1, true, NW>;
        case 2: return decode_mma_kernel<D, 2, true, NW>;
        case 3: return decode_mma_kernel<D, 3, true, NW>;
        case 4: return decode_mma_kernel<D, 4, true, NW>;
        case 5: return decode_mma_kernel<D, 5, true, NW>;
        default: return decode_mma_kernel<D, 6, true, NW>;
      }
    } else {
      switch (nbuf) {
        case 1: return decode_mma_kernel<D, 1, false, NW>;
        case 2: return decode_mma_kernel<D, 2, false, NW>;
        case 3: return decode_mma_kernel<D, 3, false, NW>;
        default: return decode_mma_kernel<D, 4, false, NW>;
      }
    }
  }
};

template <int D, bool FP8>
cudaError_t launch_mma_d(const DecodeArgs &a0, cudaStream_t s) {
  DecodeArgs a = a0;
  const int R = (a.H_q / a.H_kv) * a.T_q;
  const int fix_cap = std::min(a.n_sink, a.T_max) + std::min(a.n_stream, a.T_max);
  // keys per CTA for a cluster of C CTAs (whole 16-key sub-tiles, so a sub-tile never
  // reaches past its position array), the ring depth that holds a CTA's selected keys
  // (or its fixed ones) in one round (capped), the kernel and its shared memory
  auto shape_for = [&](const MmaShape &sh, void (**kern)(DecodeArgs), size_t *smem) {
    a.n_split = sh.C;
    auto round_up = [](int x) { return ((x + kST - 1) / kST) * kST; };
    a.sel_per = round_up((a.max_sel + sh.C - 1) / sh.C);
    a.fix_per = round_up((fix_cap + sh.C - 1) / sh.C);
    auto per_warp = [&](int keys) { return ((keys + kST - 1) / kST + sh.nw - 1) / sh.nw; };
    const int nbuf = std::min(std::max(std::max(per_warp(a.sel_per), per_warp(a.fix_per)), 1), sh.cap);
    const size_t pos = static_cast<size_t>(a.fix_per + a.sel_per) * 4;
    if (sh.nw == 8) {
      *kern = MmaKernels<D, FP8, 8>::get(nbuf);
      *smem = MmaSmem<D, FP8, 8>::rings_or_parts(nbuf, R) + pos;
    } else {
      *kern = MmaKernels<D, FP8, 4>::get(nbuf);
      *smem = MmaSmem<D, FP8, 4>::rings_or_parts(nbuf, R) + pos;
    }
  };
  cudaLaunchConfig_t cfg = {};
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the selection's last kernel runs (grid_dep_wait in the kernel)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  auto prepare = [&](const MmaShape &sh, void (**kern)(DecodeArgs)) -> cudaError_t {
    size_t smem;
    shape_for(sh, kern, &smem);
    cudaError_t e = cudaFuncSetAttribute(*kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && sh.C > 8)
      e = cudaFuncSetAttribute(*kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cfg.gridDim = dim3(sh.C, a.H_kv, a.B);
    cfg.blockDim = dim3(sh.nw * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    attr[0].val.clusterDim.x = sh.C;
    return e;
  };
  // Candidates, best first.  Eight warps with two ring slots consume a 1M-context
  // range's selected sub-tiles in one round, but their 128 KB of ring (like four warps
  // with four slots) leaves one CTA per SM: they are taken only when every cluster of
  // the launch fits the GPU at once.  Otherwise four warps with three slots (two CTAs
  // per SM); clusters of 8 where 16-CTA clusters cannot be co-scheduled at all.
  const int C0 = a.n_split;
  MmaShape cands[5];
  int n_c = 0;
  if (!FP8) cands[n_c++] = {8, C0, kMaxBuf8W};
  cands[n_c++] = {4, C0, FP8 ? kMaxBuf8 : kMaxBuf};
  if (!FP8) cands[n_c++] = {4, C0, 3};
  if (C0 > 8) cands[n_c++] = {4, 8, FP8 ? kMaxBuf8 : 3};
  const int want = a.B * a.H_kv;   // clusters of the launch
  int pick = -1, fallback = -1;
  for (int i = 0; i < n_c && pick < 0; ++i) {
    void (*kern)(DecodeArgs);
    if (prepare(cands[i], &kern) != cudaSuccess) {
      (void)cudaGetLastError();
      continue;
    }
    cfg.numAttrs = 1;   // the occupancy query sees the cluster shape only
    int n_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&n_clusters, kern, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      continue;
    }
    if (n_clusters >= want) pick = i;
    else if (n_clusters >= 1 && fallback < 0 && cands[i].nw == 4) fallback = i;
  }
  if (pick < 0) pick = fallback >= 0 ? fallback : n_c - 1;
  void (*kern)(DecodeArgs);
  cudaError_t e = prepare(cands[pick], &kern);
  if (e != cudaSuccess) return e;
  cfg.numAttrs = 2;
  {
    ProfScope ps(FP8 ? "decode_cluster_mma_fp8" : "decode_cluster_mma", s);
    e = cudaLaunchKernelEx(&cfg, kern, a);
  }
  return e;
}

}  // namespace

cudaError_t launch_decode_mma(const DecodeArgs &a, cudaStream_t s) {
  if (a.dtype == DSA_BF16_FP8KV) return launch_mma_d<128, true>(a, s);   // D = 128 checked by the API
  return a.D == 128 ? launch_mma_d<128, false>(a, s) : launch_mma_d<64, false>(a, s);
}

}  // namespace dsa
