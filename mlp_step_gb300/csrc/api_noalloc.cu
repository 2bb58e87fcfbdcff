// softmax_xent_fwd_bwd_noalloc: the softmax cross-entropy entry point for
// callers that cannot allocate device memory.  Its only scratch (the per-block
// partial losses of the fixed-order mean) lives in a file-scope device array
// of a fixed size instead of a caller-provided workspace.
#include <mutex>

#include "kernels.cuh"

namespace {

// Partial sums of the batch mean (as many floats as launch_xent's workspace
// for the batch: one per 8 rows on the multi-block path).
constexpr int kMaxPartials = 65536;  // 256 KiB
static __device__ __align__(256) float g_xent_scratch[kMaxPartials];

// Largest batch whose loss scratch fits g_xent_scratch, from the same
// workspace function the workspace entry point uses (monotone in the batch).
int max_batch() {
  int lo = 0, hi = 1 << 30;
  while (lo < hi) {
    const int mid = lo + (hi - lo + 1) / 2;
    if (mlp::xent_workspace_bytes(mid) <= sizeof(g_xent_scratch)) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Device address of g_xent_scratch on the current device.  Host code only
// sees a host-side stand-in under the array's name, so the address is looked
// up with cudaGetSymbolAddress (the device must be current) on the first call
// on each device and kept for the life of the process; after a device reset
// (cudaDeviceReset) the kept address is no longer valid.
float* scratch_address(mlp_status* st) {
  static float* addr[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *st = MLP_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_xent_scratch) != cudaSuccess || !p) {
      *st = MLP_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = static_cast<float*>(p);
  }
  *st = MLP_OK;
  return addr[dev];
}

}  // namespace

extern "C" {

int softmax_xent_noalloc_max_batch(void) {
  static const int b = max_batch();
  return b;
}

mlp_status softmax_xent_fwd_bwd_noalloc(const float* logits, int ld_logits,
                                        const int32_t* labels, int batch, int classes,
                                        float* loss_out, void* dlogits, int dlogits_dtype,
                                        int ld_dlogits, int32_t* argmax_out, void* stream) {
  if (batch < 0 || classes <= 0) return MLP_ERR_INVALID_ARG;
  if (batch == 0) return MLP_OK;
  if (mlp::xent_workspace_bytes(batch) > sizeof(g_xent_scratch)) return MLP_ERR_UNSUPPORTED_SHAPE;
  if (!logits || !labels || ld_logits < classes) return MLP_ERR_INVALID_ARG;
  if (dlogits && (ld_dlogits < classes ||
                  (dlogits_dtype != MLP_DTYPE_F32 && dlogits_dtype != MLP_DTYPE_BF16 &&
                   dlogits_dtype != MLP_DTYPE_F16)))
    return MLP_ERR_INVALID_ARG;
  if (!mlp::aligned16(logits) || !mlp::aligned16(labels) ||
      (dlogits && !mlp::aligned16(dlogits)) || (argmax_out && !mlp::aligned16(argmax_out)) ||
      (loss_out && !mlp::aligned16(loss_out)))
    return MLP_ERR_MISALIGNED;
  mlp_status st = MLP_OK;
  float* scratch = scratch_address(&st);
  if (!scratch) return st;
  // Every partial the mean reads is written by this call first, so nothing
  // has to be cleared between calls.
  return mlp::launch_xent(logits, ld_logits, labels, batch, classes, loss_out, dlogits,
                          dlogits ? dlogits_dtype : MLP_DTYPE_F32, ld_dlogits, argmax_out,
                          scratch,
                          static_cast<cudaStream_t>(stream));
}

}  // extern "C"
