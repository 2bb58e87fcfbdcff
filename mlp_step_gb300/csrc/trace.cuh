// Launch accounting and optional per-kernel timing.  Every launcher opens a
// LaunchScope around its kernel launch: the scope counts the launch and, when
// timing is enabled (eager streams only; never under stream capture),
// brackets it with CUDA events on the launching stream.
#pragma once

#include <cuda_runtime.h>

namespace mlp {

class LaunchScope {
 public:
  // `what` names the kernel; a, b, c are shape fields recorded with it
  // (for GEMMs: M, N, K).
  LaunchScope(const char* what, cudaStream_t st, long long a = 0, long long b = 0,
              long long c = 0);
  ~LaunchScope();
  LaunchScope(const LaunchScope&) = delete;
  LaunchScope& operator=(const LaunchScope&) = delete;

 private:
  cudaStream_t st_;
  int slot_;
};

}  // namespace mlp
