// sparse_attn_decode_noalloc: the split-K sparse decode with its scratch in a fixed
// device array that lives inside this library, for callers that cannot allocate
// device memory at the point of the call.
//
// Who needs it: a caller that owns no device allocator (a plain C inference engine
// or a plug-in hosted by another process's runtime), or one that must not call
// cudaMalloc on this path because cudaMalloc can synchronise the whole device and has
// no latency bound (a real-time decode loop, code running while another component
// captures work into a CUDA graph).  Such a caller still passes every input and
// output buffer; only the split-K partials move into the library's own array.
//
// The array is a file-scope __device__ variable, so every GPU that loads the library
// holds kDecodeStaticScratchBytes of it until the process exits.  Host code must not
// hand the array's name to a kernel (on the host it is only a stand-in symbol);
// the first call on each device looks up the device address with
// cudaGetSymbolAddress while that device is current and caches it.
#include <cmath>
#include <mutex>

#include "api_common.h"
#include "launch.h"

namespace dsa {
namespace {

constexpr size_t kDecodeStaticScratchBytes = size_t(4) << 20;   // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_decode_scratch[kDecodeStaticScratchBytes / sizeof(float)];

std::mutex g_scratch_mu;
float *g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device (looked up once per device).
int static_scratch(float **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(DSA_ERR_INVALID_ARG, "device ordinal %d outside [0, %d)", dev, kMaxDevices);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the static decode scratch");
    g_scratch_ptr[dev] = static_cast<float *>(p);
  }
  *out = g_scratch_ptr[dev];
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

int sparse_attn_decode_noalloc(const void *q, const void *k, const void *v,
                               const int32_t *kv_len, const int32_t *sel_idx,
                               const int32_t *sel_cnt, int max_sel, int n_sink, int n_stream,
                               float scale, const dsa_decode_shape *shape, void *out, float *lse,
                               void *stream) {
  size_t need = 0;
  // validates the shape and sizes and gives the scratch the call needs
  int st = sparse_attn_decode_workspace(shape, max_sel, n_sink, n_stream, &need);
  if (st) return st;
  if (need > kDecodeStaticScratchBytes)
    return fail(DSA_ERR_WORKSPACE,
                "this decode needs %zu bytes of scratch but the built-in array holds %zu; "
                "call sparse_attn_decode with a caller-owned workspace instead",
                need, kDecodeStaticScratchBytes);
  if (!std::isfinite(scale)) return fail(DSA_ERR_INVALID_ARG, "scale is not finite");
  const int R = (shape->H_q / shape->H_kv) * shape->T_q;
  if (R * shape->D > 4096)
    return fail(DSA_ERR_UNSUPPORTED, "(H_q/H_kv)*T_q*D = %d > 4096 rows*dims per KV head", R * shape->D);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return fail(DSA_ERR_ALIGNMENT, "q, k, v and out must be non-NULL and 16-byte aligned");
  if (!aligned(kv_len, 4) || !aligned(sel_cnt, 4) || (max_sel > 0 && !aligned(sel_idx, 4)))
    return fail(DSA_ERR_ALIGNMENT, "kv_len, sel_idx and sel_cnt must be non-NULL and 4-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(DSA_ERR_ALIGNMENT, "lse must be 4-byte aligned");
  float *part = nullptr;
  if ((st = static_scratch(&part))) return st;
  const long a_max = static_cast<long>(n_sink < shape->T_max ? n_sink : shape->T_max) + max_sel +
                     (n_stream < shape->T_max ? n_stream : shape->T_max);
  const DecodePlan plan = decode_plan(shape->B, shape->H_kv, R, shape->D, shape->dtype, static_cast<int>(a_max));
  DecodeArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.kv_len = kv_len;
  a.sel_idx = sel_idx;
  a.sel_cnt = sel_cnt;
  a.max_sel = max_sel;
  a.n_sink = n_sink;
  a.n_stream = n_stream;
  a.scale = scale;
  a.B = shape->B;
  a.T_max = shape->T_max;
  a.T_q = shape->T_q;
  a.H_q = shape->H_q;
  a.H_kv = shape->H_kv;
  a.D = shape->D;
  a.dtype = shape->dtype;
  a.n_split = plan.n_split;
  a.keys_per_split = plan.keys_per_split;
  a.cluster = plan.cluster;
  a.part = part;
  a.out = out;
  a.lse = lse;
  cudaError_t e = launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return DSA_OK;
}

}  // extern "C"
