// Device helpers shared by the kernels of libdsa (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

// Checked builds (-DDSA_CHECKS=1): a kernel that meets device-side input outside its
// documented range (a length, a count, a selected position, a list entry) still skips
// or clamps it as the normal build does, and also records the fact in a check word of
// its translation unit; dsa_device_error reports any of them as DSA_ERR_DEVICE_CHECK.
// DSA_CHECK_WORD(name) defines the word and a host reader `int name()` (read and
// clear; -1 on a CUDA error; always 0 in normal builds).
#ifndef DSA_CHECKS
#define DSA_CHECKS 0
#endif
#if DSA_CHECKS
#define DSA_CHECK(cond)                                  \
  do {                                                   \
    if (!(cond)) atomicOr(&g_dsa_check_word, 1);         \
  } while (0)
#define DSA_CHECK_WORD(name)                                                         \
  static __device__ int g_dsa_check_word;                                           \
  int name() {                                                                       \
    int v = 0, z = 0;                                                                \
    if (cudaMemcpyFromSymbol(&v, g_dsa_check_word, sizeof(int)) != cudaSuccess) return -1; \
    if (cudaMemcpyToSymbol(g_dsa_check_word, &z, sizeof(int)) != cudaSuccess) return -1;   \
    return v;                                                                        \
  }
#else
#define DSA_CHECK(cond) \
  do {                  \
  } while (0)
#define DSA_CHECK_WORD(name) \
  int name() { return 0; }
#endif

namespace dsa {

constexpr unsigned kFull = 0xffffffffu;

// Programmatic dependent launch: a kernel launched with launch_pdl may be scheduled
// while the previous kernel of the stream drains; it must call grid_dep_wait() before
// it reads anything an earlier kernel wrote or writes anything an earlier kernel
// reads.  A kernel launched the ordinary way returns from it at once.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
// Lets the next kernel of the stream (launched with launch_pdl or the same attribute)
// start before this one finishes; it still waits in grid_dep_wait() for this grid's
// results.
__device__ __forceinline__ void grid_dep_release() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// fp32 -> bf16 bits, round to nearest even (inputs here are finite).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// Unpack 16 bytes of storage into floats: 8 bf16 or 4 fp32.
__device__ __forceinline__ void unpack16(const uint4 &u, float *f, uint16_t) {
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
  f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
  f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}
__device__ __forceinline__ void unpack16(const uint4 &u, float *f, float) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}

// Storage tag of FP8 E4M3 key / value rows (one byte per element).
struct Fp8E4M3 {
  uint8_t bits;
};

// One FP8 E4M3 code -> float, exactly.  E4M3 is sign, 4 exponent bits (bias 7) and 3
// mantissa bits; placed in the top of an fp32's exponent/mantissa fields they read as
// the same value times 2^-120 (a normal code becomes a normal fp32, a subnormal one a
// subnormal fp32, both exact), so one multiply by 2^120 restores it.  Inputs are never
// the NaN code.
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  const float mag = __uint_as_float((c & 0x7Fu) << 20) * 0x1p120f;
  return (c & 0x80u) ? -mag : mag;
}

__device__ __forceinline__ void unpack16(const uint4 &u, float *f, Fp8E4M3) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int b = 0; b < 4; ++b) f[4 * i + b] = e4m3_to_f32((w[i] >> (8 * b)) & 0xFFu);
  }
}

template <typename T> struct Store;
template <> struct Store<uint16_t> { static constexpr int kPer16 = 8; };
template <> struct Store<float> { static constexpr int kPer16 = 4; };
template <> struct Store<Fp8E4M3> { static constexpr int kPer16 = 16; };

// Load N consecutive elements (N * sizeof(T) a multiple of 16, 16-byte aligned) as floats.
template <typename T, int N>
__device__ __forceinline__ void load_row(const T *p, float *f) {
  constexpr int per = Store<T>::kPer16;
  const uint4 *p4 = reinterpret_cast<const uint4 *>(p);
#pragma unroll
  for (int i = 0; i < N / per; ++i) {
    uint4 u = __ldg(p4 + i);
    unpack16(u, f + i * per, T());
  }
}

// Monotone map float -> uint32 (larger float -> larger key); -0 == +0; NaN lowest.
__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) == 0u) u = 0u;
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// Block-wide radix select: the K-th largest of n 32-bit keys (1 <= K <= n).
// key_of(i) must return the same key every time it is called for i.
// Result: thr = that key; k_eq = how many elements equal to thr belong to the
// top K (so K - k_eq elements are strictly larger).  All threads get both.
// s_hist: 256 words of shared memory; s_res: 2 words.
// ---------------------------------------------------------------------------
template <int NT, typename KeyFn>
__device__ void block_radix_select(KeyFn key_of, int n, int K, uint32_t *s_hist,
                                   uint32_t *s_res, uint32_t &thr, int &k_eq) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0, mask = 0;
  uint32_t k_rem = static_cast<uint32_t>(K);
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += NT) s_hist[i] = 0;
    __syncthreads();
    // uniform trip count over the block; lanes with the same bin add once together
    for (int i0 = 0; i0 < n; i0 += NT) {
      const int i = i0 + tid;
      const uint32_t kk = i < n ? key_of(i) : 0u;
      const bool ok = i < n && (kk & mask) == prefix;
      const uint32_t bin = ok ? ((kk >> shift) & 255u) : 256u;
      const unsigned peers = __match_any_sync(kFull, bin);
      if (ok && lane == __ffs(peers) - 1) atomicAdd(&s_hist[bin], static_cast<uint32_t>(__popc(peers)));
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255-8l .. 248-8l, scanned from the top down
      const int top = 255 - lane * 8;
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int t = 0; t < 8; ++t) { c[t] = s_hist[top - t]; sum += c[t]; }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
      }
      uint32_t excl = incl - sum;
      if (excl < k_rem && k_rem <= incl) {
        uint32_t run = excl;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (run + c[t] >= k_rem) { s_res[0] = static_cast<uint32_t>(top - t); s_res[1] = run; break; }
          run += c[t];
        }
      }
    }
    __syncthreads();
    const uint32_t digit = s_res[0], above = s_res[1];
    prefix |= digit << shift;
    mask |= 255u << shift;
    k_rem -= above;
    __syncthreads();
  }
  thr = prefix;
  k_eq = static_cast<int>(k_rem);
}

// Block-wide exclusive scan of one flag per thread over a tile of NT elements.
// Returns this thread's rank among set flags in the tile; *total = tile count.
// s_warp: NT/32 + 1 words of shared memory.  All threads must call it.
template <int NT>
__device__ __forceinline__ int block_flag_rank(bool f, int *s_warp, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = NT / 32;
  unsigned bal = __ballot_sync(kFull, f);
  int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) s_warp[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    int v = lane < NW ? s_warp[lane] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane < NW) s_warp[lane] = incl - v;
    if (lane == 31) s_warp[NW] = incl;
  }
  __syncthreads();
  int r = s_warp[warp] + in_warp;
  *total = s_warp[NW];
  __syncthreads();
  return r;
}

}  // namespace dsa
