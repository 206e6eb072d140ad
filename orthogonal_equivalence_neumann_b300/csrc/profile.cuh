// profile.cuh -- per-launch accounting used by every kernel launcher.
#pragma once

#include <cuda_runtime.h>

namespace poetx {

// Construct immediately before a kernel launch and let it go out of scope
// right after it: counts the launch and, while profiling is on, records a
// CUDA event before and after it on the same stream.
class KernelScope {
 public:
  KernelScope(const char* name, cudaStream_t s);
  ~KernelScope();
  KernelScope(const KernelScope&) = delete;
  KernelScope& operator=(const KernelScope&) = delete;

 private:
  const char* name_;
  cudaStream_t stream_;
  cudaEvent_t begin_ = nullptr, end_ = nullptr;
};

}  // namespace poetx
