// Error reporting and version entry points of the C ABI.
#include "api_common.h"

#include <cstring>

namespace dsa {

namespace {
thread_local char g_msg[512] = "";
}

const char *last_error() { return g_msg; }

void clear_error() { g_msg[0] = '\0'; }

int fail(int status, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char *what) {
  return fail(DSA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

}  // namespace dsa

extern "C" {

const char *dsa_last_error(void) { return dsa::last_error(); }

const char *dsa_strerror(int status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case DSA_ERR_WORKSPACE: return "workspace missing or too small";
    case DSA_ERR_ALIGNMENT: return "null or misaligned pointer";
    case DSA_ERR_CUDA: return "CUDA launch error";
    case DSA_ERR_DEVICE_CHECK: return "device-side check failed";
    default: return "unknown status";
  }
}

int dsa_version(void) { return DSA_VERSION; }

}  // extern "C"
