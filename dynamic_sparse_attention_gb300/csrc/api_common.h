// Host-side helpers of the C-ABI layer: error reporting, alignment checks and
// workspace carving.  Internal to libdsa.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>

#include "dsa.h"

namespace dsa {

// thread-local message of the last failure (set by fail())
const char *last_error();
int fail(int status, const char *fmt, ...);
int cuda_fail(cudaError_t e, const char *what);
void clear_error();

inline bool aligned(const void *p, size_t a) {
  return p != nullptr && (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Bump allocator over the caller's workspace; every piece is 256-byte aligned.
struct Carve {
  char *base;
  size_t off = 0;
  explicit Carve(void *b) : base(static_cast<char *>(b)) {}
  template <typename T>
  T *take(size_t n) {
    off = (off + 255) & ~size_t(255);
    T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
    off += n * sizeof(T);
    return p;
  }
  size_t bytes() const { return (off + 255) & ~size_t(255); }
};

}  // namespace dsa
