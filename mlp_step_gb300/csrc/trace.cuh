// Launch accounting and optional per-kernel timing.  Every launcher opens a
// LaunchScope around its kernel launch: the scope counts the launch and, when
// timing is enabled (eager streams only; never under stream capture),
// brackets it with CUDA events on the launching stream.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

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

// A named NVTX range over one library call (a training step, an epoch, a
// block pass), so that a timeline profiler groups each call's kernels under
// its name.  NVTX3 is header-only; without a profiler attached the push and
// pop cost a branch.
class NvtxRange {
 public:
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace mlp
