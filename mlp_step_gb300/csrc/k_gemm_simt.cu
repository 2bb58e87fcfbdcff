// fp32 SIMT GEMM with the fused epilogue: the fp32 path of the 784-256-10
// step ("The Work Moved Down a Layer", "Cooperation Beats Isolation": an fp32
// route beside the matrix-unit route) and the K = 0 case of the bf16 path.
//
// "Capstone 5: train a network with your CUDA kernels", "Read the worked
// reference": the multiply keeps bias and ReLU in its epilogue and writes no
// separate bias or ReLU array; "Work through the backward pass": the weight
// and input gradients read one operand transposed, here by indexing the
// operand tile loads, never by a transpose copy.
//
// 64x64 output tile per block, 256 threads each owning a 4x4 micro-tile, K in
// steps of 16 staged through shared memory.  Each output sums k in ascending
// order, so the result is deterministic.
#include "kernels.cuh"
#include "trace.cuh"

namespace mlp {

template <typename T>
__device__ __forceinline__ float ld_in(const T* p);
template <>
__device__ __forceinline__ float ld_in<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_in<__nv_bfloat16>(const __nv_bfloat16* p) {
  return bf16_to_f32(*p);
}

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs g) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const T* A = static_cast<const T*>(g.A);
  const T* B = static_cast<const T*>(g.B);
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};

  for (int k0 = 0; k0 < g.K; k0 += 16) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int idx = tid + e * 256;
      int m, k;
      if (!g.a_trans) { m = idx >> 4; k = idx & 15; }
      else { k = idx >> 6; m = idx & 63; }
      const int gm = m0 + m, gk = k0 + k;
      float v = 0.f;
      if (gm < g.M && gk < g.K)
        v = g.a_trans ? ld_in(A + (size_t)gk * g.lda + gm) : ld_in(A + (size_t)gm * g.lda + gk);
      As[k][m] = v;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int idx = tid + e * 256;
      int n, k;
      if (!g.b_trans) { k = idx >> 6; n = idx & 63; }
      else { n = idx >> 4; k = idx & 15; }
      const int gn = n0 + n, gk = k0 + k;
      float v = 0.f;
      if (gn < g.N && gk < g.K)
        v = g.b_trans ? ld_in(B + (size_t)gn * g.ldb + gk) : ld_in(B + (size_t)gk * g.ldb + gn);
      Bs[k][n] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] += a[i] * b[j];
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= g.N) continue;
      float v = acc[i][j];
      if (g.bias) v += g.bias[n];
      if (g.act == MLP_ACT_RELU) v = fmaxf(v, 0.f);
      if (g.mask) {
        const float mk = ld_in(static_cast<const T*>(g.mask) + (size_t)m * g.ldm + n);
        v = mk > 0.f ? v : 0.f;
      }
      if (g.c_bf16) static_cast<__nv_bfloat16*>(g.C)[(size_t)m * g.ldc + n] = f32_to_bf16(v);
      else static_cast<float*>(g.C)[(size_t)m * g.ldc + n] = v;
    }
  }
}

mlp_status launch_gemm_simt(const GemmArgs& g, int in_bf16, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0) return MLP_OK;
  dim3 grid((g.N + 63) / 64, (g.M + 63) / 64);
  if (grid.y > 65535) return MLP_ERR_UNSUPPORTED_SHAPE;
  LaunchScope ls("gemm_simt", st, g.M, g.N, g.K);
  if (in_bf16) launch_k(gemm_simt_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, st, g);
  else launch_k(gemm_simt_kernel<float>, dim3(grid), dim3(256), 0, st, g);
  return launch_status();
}

}  // namespace mlp
