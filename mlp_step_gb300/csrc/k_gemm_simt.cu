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
// order, so the result is deterministic.  For fp32 operands the K steps
// stream through a 4-deep ring of cp.async copies (zero-filled past the
// edges), so a block waits on one global-memory round trip per four steps
// rather than per step: at the batch sizes of the minimum model the grid has
// a handful of blocks and the loop is latency-bound.
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
      // 16-bit outputs in the operands' format (fp16 when g.f16 is set)
      if (g.c_bf16)
        static_cast<uint16_t*>(g.C)[(size_t)m * g.ldc + n] =
            f32_to_16_fmt(v, g.f16 ? MLP_DTYPE_F16 : MLP_DTYPE_BF16);
      else static_cast<float*>(g.C)[(size_t)m * g.ldc + n] = v;
    }
  }
}

constexpr int SIMT_STAGES = 4;
constexpr int SIMT_SLOT = 64 * 20;  // floats per operand slot: [64][16 + 4] or [16][64 + 4]

__device__ __forceinline__ void cp_async_f32(float* smem_dst, const float* src, bool valid) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  // src-size 0 writes zeros (and reads nothing) for elements past the edges
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(d), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}

__device__ __forceinline__ void cp_async_16(float* smem_dst, const float* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}

// Four consecutive elements of a row of a row-major operand (row `r`, column
// `c0`, leading dimension ld) into 16 contiguous bytes of shared memory:
// one 16-byte copy when the four are in range and aligned, else element-wise
// (zero-filled past the edges).
__device__ __forceinline__ void stage_quad(float* dst, const float* base, int ld, int r, int c0,
                                           int rows, int cols, bool vec) {
  if (vec && r < rows && c0 + 3 < cols) {
    cp_async_16(dst, base + (size_t)r * ld + c0);
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool ok = r < rows && c0 + e < cols;
      cp_async_f32(dst + e, ok ? base + (size_t)r * ld + c0 + e : base, ok);
    }
  }
}

// Split-K scratch (in the caller's workspace g.ws): per-tile arrival counters,
// then the raw 64 x 64 partial sums of every (tile, split).
constexpr int kSimtCounters = 512;
constexpr int kSimtMaxParts = 304;

__global__ void __launch_bounds__(256) gemm_simt_f32_pipelined_kernel(GemmArgs g) {
  pdl_wait();
  pdl_launch_dependents();
  // split z of gridDim.z sums k-steps [kt0, kt1); with splits the last split
  // of a tile to finish adds the partials in split order (deterministic) and
  // runs the epilogue
  const int splits = gridDim.z, z = blockIdx.z;
  __shared__ int s_last;
  // A slot: [64 m][20] (A stored [M][K]) or [16 k][68] (stored [K][M]);
  // B slot: [16 k][68] (B stored [K][N]) or [64 n][20] (stored [N][K]).
  __shared__ __align__(16) float As[SIMT_STAGES][SIMT_SLOT];
  __shared__ __align__(16) float Bs[SIMT_STAGES][SIMT_SLOT];
  const float* A = static_cast<const float*>(g.A);
  const float* B = static_cast<const float*>(g.B);
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int nk_all = (g.K + 15) / 16;
  const int per = (nk_all + splits - 1) / splits;
  const int kt0 = z * per < nk_all ? z * per : nk_all;
  const int nk = (kt0 + per < nk_all ? kt0 + per : nk_all) - kt0;  // k-steps of this split
  const bool a_vec = (reinterpret_cast<uintptr_t>(A) & 15) == 0 && (g.lda & 3) == 0;
  const bool b_vec = (reinterpret_cast<uintptr_t>(B) & 15) == 0 && (g.ldb & 3) == 0;
  float acc[4][4] = {};

  // each thread stages one quad of each operand per step
  auto issue = [&](int kt) {
    const int st = kt % SIMT_STAGES, k0 = (kt0 + kt) * 16;
    if (!g.a_trans) {
      const int m = tid >> 2, kq = (tid & 3) * 4;
      stage_quad(&As[st][m * 20 + kq], A, g.lda, m0 + m, k0 + kq, g.M, g.K, a_vec);
    } else {
      const int k = tid >> 4, mq = (tid & 15) * 4;
      stage_quad(&As[st][k * 68 + mq], A, g.lda, k0 + k, m0 + mq, g.K, g.M, a_vec);
    }
    if (!g.b_trans) {
      const int k = tid >> 4, nq = (tid & 15) * 4;
      stage_quad(&Bs[st][k * 68 + nq], B, g.ldb, k0 + k, n0 + nq, g.K, g.N, b_vec);
    } else {
      const int n = tid >> 2, kq = (tid & 3) * 4;
      stage_quad(&Bs[st][n * 20 + kq], B, g.ldb, n0 + n, k0 + kq, g.N, g.K, b_vec);
    }
  };

  // prologue: the first STAGES - 1 steps in flight (one commit group each,
  // empty groups past the end keep the group count uniform)
#pragma unroll
  for (int kt = 0; kt < SIMT_STAGES - 1; ++kt) {
    if (kt < nk) issue(kt);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int kt = 0; kt < nk; ++kt) {
    // step kt has landed once at most STAGES - 2 newer groups are pending
    asm volatile("cp.async.wait_group %0;" ::"n"(SIMT_STAGES - 2) : "memory");
    __syncthreads();
    // refill the slot the previous step used (all threads are past it)
    if (kt + SIMT_STAGES - 1 < nk) issue(kt + SIMT_STAGES - 1);
    asm volatile("cp.async.commit_group;" ::: "memory");
    const float* as = As[kt % SIMT_STAGES];
    const float* bs = Bs[kt % SIMT_STAGES];
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        a[i] = g.a_trans ? as[kk * 68 + ty * 4 + i] : as[(ty * 4 + i) * 20 + kk];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        b[j] = g.b_trans ? bs[(tx * 4 + j) * 20 + kk] : bs[kk * 68 + tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] += a[i] * b[j];
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");

  if (splits > 1) {
    const int tile = blockIdx.y * gridDim.x + blockIdx.x;
    unsigned* counters = static_cast<unsigned*>(g.ws);
    float* parts = reinterpret_cast<float*>(static_cast<uint8_t*>(g.ws) + kSimtCounters * 4);
    float* mine = parts + ((size_t)tile * splits + z) * 4096;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(mine + (ty * 4 + i) * 64 + tx * 4) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&counters[tile], 1u) == (unsigned)(splits - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int z2 = 0; z2 < splits; ++z2) {
      const float* pz = parts + ((size_t)tile * splits + z2) * 4096;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 q = __ldcg(reinterpret_cast<const float4*>(pz + (ty * 4 + i) * 64 + tx * 4));
        acc[i][0] += q.x; acc[i][1] += q.y; acc[i][2] += q.z; acc[i][3] += q.w;
      }
    }
    if (tid == 0) counters[tile] = 0;  // ready for the next launch
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
        const float mk = ld_in(static_cast<const float*>(g.mask) + (size_t)m * g.ldm + n);
        v = mk > 0.f ? v : 0.f;
      }
      if (g.c_bf16) static_cast<__nv_bfloat16*>(g.C)[(size_t)m * g.ldc + n] = f32_to_bf16(v);
      else static_cast<float*>(g.C)[(size_t)m * g.ldc + n] = v;
    }
  }
}

size_t gemm_simt_scratch_bytes() {
  return (size_t)kSimtCounters * 4 + (size_t)kSimtMaxParts * 64 * 64 * 4;
}

// K splits of an fp32 GEMM: when its tiles leave most SMs idle, K is cut so
// that about one CTA per SM runs (each split at least two 16-deep steps);
// needs the split-K scratch in g.ws (counters zero between launches).  Never
// in the linear-order mode.
static int simt_splits(const GemmArgs& g, int tiles) {
  if (linear_order()) return 1;  // one FMA chain over all of K per output
  if (!g.ws || g.ws_bytes < gemm_simt_scratch_bytes() || (reinterpret_cast<uintptr_t>(g.ws) & 15))
    return 1;
  if (tiles >= num_sms() || tiles > kSimtCounters) return 1;
  const int nk = (g.K + 15) / 16;
  int s = (num_sms() + tiles - 1) / tiles;
  if (s > nk / 2) s = nk / 2;
  if (s * tiles > kSimtMaxParts) s = kSimtMaxParts / tiles;
  return s < 1 ? 1 : s;
}

mlp_status launch_gemm_simt(const GemmArgs& g, int in_bf16, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0) return MLP_OK;
  dim3 grid((g.N + 63) / 64, (g.M + 63) / 64);
  if (grid.y > 65535) return MLP_ERR_UNSUPPORTED_SHAPE;
  LaunchScope ls("gemm_simt", st, g.M, g.N, g.K);
  if (in_bf16) {
    launch_k(gemm_simt_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, st, g);
  } else {
    grid.z = simt_splits(g, (int)(grid.x * grid.y));
    launch_k(gemm_simt_f32_pipelined_kernel, dim3(grid), dim3(256), 0, st, g);
  }
  return launch_status();
}

}  // namespace mlp
