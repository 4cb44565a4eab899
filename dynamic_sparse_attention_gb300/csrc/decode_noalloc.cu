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
// cudaGetSymbolAddress while that device is current and caches it for that device's
// context.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "api_common.h"
#include "launch.h"

namespace dsa {
namespace {

constexpr size_t kDecodeStaticScratchBytes = size_t(4) << 20;   // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_decode_scratch[kDecodeStaticScratchBytes / sizeof(float)];

std::mutex g_scratch_mu;

// The address is valid for one CUDA context: a cudaDeviceReset (by the host program or
// another library) destroys the primary context and unloads this module's copy of the
// array, and the next context may place it elsewhere.  So each device's cached address
// is tagged with the unique id of the context it was looked up in (cuCtxGetId) and
// looked up again when the current context's id differs.
struct ScratchSlot {
  unsigned long long ctx_id;
  float *ptr;
};
ScratchSlot g_slot[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// id of the calling thread's current context; false if there is none or the driver
// does not say
bool current_ctx_id(unsigned long long *id) {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_cur || !get_id) return false;
  CUcontext c = nullptr;
  if (get_cur(&c) != CUDA_SUCCESS || c == nullptr) return false;
  return get_id(c, id) == CUDA_SUCCESS;
}

// Device address of the array in the current device's current context: looked up with
// cudaGetSymbolAddress on the first call in a context, cached after that.
int static_scratch(float **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(DSA_ERR_INVALID_ARG, "device ordinal %d outside [0, %d)", dev, kMaxDevices);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  unsigned long long id = 0;
  if (g_slot[dev].ptr && current_ctx_id(&id) && id == g_slot[dev].ctx_id) {
    *out = g_slot[dev].ptr;
    return DSA_OK;
  }
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_decode_scratch);   // also makes the primary context current
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the static decode scratch");
  g_slot[dev].ptr = static_cast<float *>(p);
  g_slot[dev].ctx_id = current_ctx_id(&id) ? id : 0ull;   // 0: not cached, look up next time
  if (!g_slot[dev].ctx_id) g_slot[dev].ptr = nullptr;
  *out = static_cast<float *>(p);
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
  clear_error();
  DecodeArgs a{};
  size_t nf = 0;
  // the same checks and arguments as sparse_attn_decode; only the partials differ
  int st = decode_prepare(q, k, v, kv_len, sel_idx, sel_cnt, max_sel, n_sink, n_stream, scale,
                          shape, out, lse, &a, &nf);
  if (st) return st;
  Carve cv(nullptr);
  if (nf) cv.take<float>(nf);
  if (cv.bytes() > kDecodeStaticScratchBytes)
    return fail(DSA_ERR_WORKSPACE,
                "this decode needs %zu bytes of scratch but the built-in array holds %zu; "
                "call sparse_attn_decode with a caller-owned workspace instead",
                cv.bytes(), kDecodeStaticScratchBytes);
  if (nf && (st = static_scratch(&a.part))) return st;
  cudaError_t e = launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return DSA_OK;
}

}  // extern "C"
