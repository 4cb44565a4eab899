// Opt-in per-kernel CUDA-event timing and its C entry points.
#include "profile.h"

#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "api_common.h"

namespace dsa {
namespace {

struct Rec {
  const char *name;
  cudaEvent_t a, b;
};

std::atomic<bool> g_on{false};
std::mutex g_mu;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

ProfScope::ProfScope(const char *name, cudaStream_t s) : name_(name), s_(s) {
  if (!g_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  a_ = take_event();
  b_ = take_event();
  if (a_ && b_) cudaEventRecord(a_, s_);
}

ProfScope::~ProfScope() {
  if (!a_ || !b_) return;
  cudaEventRecord(b_, s_);
  std::lock_guard<std::mutex> lk(g_mu);
  g_recs.push_back({name_, a_, b_});
}

}  // namespace dsa

extern "C" {

int dsa_profile_enable(int on) {
  dsa::g_on.store(on != 0);
  return DSA_OK;
}

int dsa_profile_collect(dsa_kernel_stat *out, int max_out, int *n_out) {
  using namespace dsa;
  clear_error();
  if (!n_out || (max_out > 0 && !out)) return fail(DSA_ERR_ALIGNMENT, "output pointers are NULL");
  std::lock_guard<std::mutex> lk(g_mu);
  std::vector<dsa_kernel_stat> acc;
  int status = DSA_OK;
  for (const Rec &r : g_recs) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.a, r.b);
    if (e != cudaSuccess && status == DSA_OK) status = cuda_fail(e, "profile event");
    size_t k = 0;
    while (k < acc.size() && std::strcmp(acc[k].name, r.name) != 0) ++k;
    if (k == acc.size()) acc.push_back({r.name, 0, 0.0});
    acc[k].launches += 1;
    acc[k].total_ms += ms;
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.clear();
  const int n = static_cast<int>(acc.size());
  for (int i = 0; i < n && i < max_out; ++i) out[i] = acc[i];
  *n_out = n;
  return status;
}

}  // extern "C"
