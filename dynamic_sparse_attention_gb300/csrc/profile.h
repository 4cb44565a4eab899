// Opt-in per-kernel timing: when enabled, each launch is bracketed by two CUDA
// events recorded on the launch's own stream.  Disabled (the default), a scope
// costs one relaxed atomic load.  Internal to libdsa.
#pragma once

#include <cuda_runtime.h>

namespace dsa {

class ProfScope {
 public:
  ProfScope(const char *name, cudaStream_t s);
  ~ProfScope();
  ProfScope(const ProfScope &) = delete;
  ProfScope &operator=(const ProfScope &) = delete;

 private:
  const char *name_;
  cudaStream_t s_;
  cudaEvent_t a_ = nullptr, b_ = nullptr;
};

}  // namespace dsa
