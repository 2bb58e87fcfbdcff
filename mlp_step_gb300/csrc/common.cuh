// Shared definitions of the CUDA library: status codes, the device error word,
// bf16 / fp16 helpers and launch checks.  Nothing here is used by the oracle.
#pragma once

#include <cstdint>
#include <cstddef>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/mlp_step.h"

namespace mlp {

// Device-side error word.  Kernels that give up on a bounded wait record a
// code there instead of trapping; mlp_get_device_status() reads and clears
// it.  The word lives in api.cu; kernels receive its device address.
int* device_error_word();

// Error codes written into g_device_error (high bits: where, low bits: what).
enum : int {
  DEVERR_NONE = 0,
  DEVERR_TIMEOUT_PRODUCER = 0x101,
  DEVERR_TIMEOUT_MMA = 0x102,
  DEVERR_TIMEOUT_EPILOGUE = 0x103,
  DEVERR_TIMEOUT_TEARDOWN = 0x104,
  DEVERR_TIMEOUT_PEER = 0x105,
  DEVERR_TIMEOUT_GRID = 0x106,
  DEVERR_NUMERIC = 0x201,  // a loss kernel produced a non-finite loss
};

__device__ __forceinline__ void record_device_error(int* word, int code) {
  if (word) atomicCAS(word, 0, code);
}

// A loss that is not finite (an overflowing or NaN logit or output reached
// the mean) is recorded for mlp_get_device_status (MLP_ERR_NUMERIC); the value
// itself is still stored.
__device__ __forceinline__ void check_loss_finite(float loss, int* err) {
  if (!isfinite(loss)) record_device_error(err, DEVERR_NUMERIC);
}

__device__ __forceinline__ float bf16_to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ __nv_bfloat16 f32_to_bf16(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 p = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// The tensor-core path's 16-bit operand format: H16 = 0 for bf16, 1 for fp16
// (the same storage size and the same sign / zero encoding, so 16-bit
// buffers travel as raw bits and ReLU masks read either format).
template <int H16>
__device__ __forceinline__ uint32_t pack16x2(float lo, float hi) {
  if constexpr (H16) return pack_f16x2(lo, hi);
  else return pack_bf16x2(lo, hi);
}

template <int H16>
__device__ __forceinline__ uint16_t f32_to_16(float v) {
  if constexpr (H16) return __half_as_ushort(__float2half_rn(v));
  else return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// Runtime-format forms for the bandwidth-bound kernels.  fmt: MLP_DTYPE_BF16
// or MLP_DTYPE_F16.
__device__ __forceinline__ uint32_t pack16x2_fmt(float lo, float hi, int fmt) {
  return fmt == MLP_DTYPE_F16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
}

__device__ __forceinline__ uint16_t f32_to_16_fmt(float v, int fmt) {
  return fmt == MLP_DTYPE_F16 ? __half_as_ushort(__float2half_rn(v))
                              : __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float f16bits_to_f32(uint16_t b, int fmt) {
  return fmt == MLP_DTYPE_F16 ? __half2float(__ushort_as_half(b))
                              : __bfloat162float(__ushort_as_bfloat16(b));
}

// Programmatic dependent launch: kernels launched through launch_k may start
// (their prologue: barriers, tensor memory, tensor-map prefetch) while the
// previous kernel on the stream finishes; each kernel calls pdl_wait() before
// its first global-memory access, which waits for the previous grid to
// complete and its writes to be visible, and pdl_launch_dependents() so that
// the next kernel may be scheduled.  Without the launch attribute both are
// no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

bool pdl_enabled();

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

// Translate the last launch error into a status.
inline mlp_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MLP_OK : MLP_ERR_CUDA;
}

#define MLP_CHECK(expr)                      \
  do {                                       \
    mlp_status _s = (expr);                  \
    if (_s != MLP_OK) return _s;             \
  } while (0)

}  // namespace mlp
