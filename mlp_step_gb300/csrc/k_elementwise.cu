// Memory-bound kernels of the training step: momentum SGD over the flat
// parameter buffer (with the bf16 shadow refresh fused in), input casting,
// stable softmax cross entropy, column-sum bias gradients and the
// mean-squared loss.  All reductions run in fp32 with a fixed summation order,
// so results are bitwise reproducible from run to run.
#include "kernels.cuh"
#include "ptx.cuh"
#include "trace.cuh"
#include "xent_row.cuh"

namespace mlp {

// ------------------------------------------------------------------ SGD
//
// "Capstone 5: train a network with your CUDA kernels", "Read the worked
// reference": one grid-stride kernel updates every weight and velocity of the
// flat buffer: v <- m v - lr g;  w <- w + v.  Here the body moves 16 bytes per
// load/store (float4) with streaming cache hints; each element also writes
// bf16(w) into the weight shadow the tensor-core GEMMs read, through a
// per-segment map (row-padded for narrow layers).

__device__ __forceinline__ int find_segment(const SgdSegments& s, long long i) {
  int k = 0;
  while (k + 1 < s.n && i >= s.flat_off[k + 1]) ++k;
  return k;
}

__device__ __forceinline__ long long shadow_index(const SgdSegments& s, int k, long long i) {
  const long long j = i - s.flat_off[k];
  if (s.cols[k] == s.cols_pad[k]) return s.shadow_off[k] + j;
  const long long r = j / s.cols[k];
  return s.shadow_off[k] + r * s.cols_pad[k] + (j - r * s.cols[k]);
}

__device__ __forceinline__ void sgd_scalar(float* w, const float* g, float* v,
                                           uint16_t* wb, int wb_fmt, const SgdSegments& s,
                                           long long i, float lr, float mom) {
  const float vel = mom * v[i] - lr * g[i];
  const float nw = w[i] + vel;
  v[i] = vel;
  w[i] = nw;
  if (wb) {
    const int k = find_segment(s, i);
    if (s.shadow_off[k] >= 0) wb[shadow_index(s, k, i)] = f32_to_16_fmt(nw, wb_fmt);
  }
}

__global__ void __launch_bounds__(256) sgd_kernel(float* __restrict__ w, const float* __restrict__ g,
                                                  float* __restrict__ v,
                                                  uint16_t* __restrict__ wb, int wb_fmt,
                                                  long long n, float lr, float mom,
                                                  SgdSegments segs) {
  pdl_wait();
  pdl_launch_dependents();
  const long long n4 = n >> 2;
  const long long stride = (long long)gridDim.x * blockDim.x;
  float4* w4 = reinterpret_cast<float4*>(w);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  float4* v4 = reinterpret_cast<float4*>(v);
  for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < n4; q += stride) {
    const float4 gq = __ldcs(g4 + q);
    const float4 vq = __ldcs(v4 + q);
    const float4 wq = __ldcs(w4 + q);
    float4 nv, nw;
    nv.x = mom * vq.x - lr * gq.x;  nw.x = wq.x + nv.x;
    nv.y = mom * vq.y - lr * gq.y;  nw.y = wq.y + nv.y;
    nv.z = mom * vq.z - lr * gq.z;  nw.z = wq.z + nv.z;
    nv.w = mom * vq.w - lr * gq.w;  nw.w = wq.w + nv.w;
    __stcs(v4 + q, nv);
    __stcs(w4 + q, nw);
    if (wb) {
      const long long i = q << 2;
      const int k = find_segment(segs, i);
      const bool same = (k + 1 >= segs.n) || (i + 3 < segs.flat_off[k + 1]);
      // the group's shadow position when its four elements share one row
      long long si = -1;
      if (same && segs.shadow_off[k] >= 0) {
        const long long local = i - segs.flat_off[k];
        if (segs.cols[k] == segs.cols_pad[k]) {
          si = segs.shadow_off[k] + local;
        } else if (local < (1ll << 31)) {
          const unsigned cols = (unsigned)segs.cols[k];
          const unsigned r = (unsigned)local / cols, c = (unsigned)local - r * cols;
          if (c + 3 < cols) si = segs.shadow_off[k] + (long long)r * segs.cols_pad[k] + c;
        }
      }
      if (si >= 0) {
        uint2 pk;
        pk.x = pack16x2_fmt(nw.x, nw.y, wb_fmt);
        pk.y = pack16x2_fmt(nw.z, nw.w, wb_fmt);
        if ((si & 3) == 0) {
          __stcs(reinterpret_cast<uint2*>(wb + si), pk);
        } else {
          wb[si] = (uint16_t)(pk.x & 0xffffu); wb[si + 1] = (uint16_t)(pk.x >> 16);
          wb[si + 2] = (uint16_t)(pk.y & 0xffffu); wb[si + 3] = (uint16_t)(pk.y >> 16);
        }
      } else {
        const float vals[4] = {nw.x, nw.y, nw.z, nw.w};
        for (int e = 0; e < 4; ++e) {
          const int ke = find_segment(segs, i + e);
          if (segs.shadow_off[ke] >= 0)
            wb[shadow_index(segs, ke, i + e)] = f32_to_16_fmt(vals[e], wb_fmt);
        }
      }
    }
  }
  // scalar tail (n not a multiple of 4)
  const long long t = (n4 << 2) + (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t < n) sgd_scalar(w, g, v, wb, wb_fmt, segs, t, lr, mom);
}

// Shadow refresh alone: wb <- bf16(w) or fp16(w) through the segment map.
__global__ void shadow_kernel(const float* __restrict__ w, uint16_t* __restrict__ wb,
                              int wb_fmt, long long n, SgdSegments segs) {
  pdl_wait();
  pdl_launch_dependents();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int k = find_segment(segs, i);
    if (segs.shadow_off[k] >= 0) wb[shadow_index(segs, k, i)] = f32_to_16_fmt(w[i], wb_fmt);
  }
}

int sgd_grid(long long n) {
  const long long q = (n + 3) / 4;
  long long blocks = (q + 255) / 256;
  const long long cap = (long long)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

mlp_status launch_sgd(float* w, const float* g, float* v, void* wb, int wb_fmt, long long n,
                      float lr, float mom, const SgdSegments& segs, cudaStream_t st) {
  if (n <= 0) return MLP_OK;
  LaunchScope ls("sgd", st, n);
  launch_k(sgd_kernel, dim3(sgd_grid(n)), dim3(256), 0, st, w, g, v, static_cast<uint16_t*>(wb),
           wb_fmt, n, lr, mom, segs);
  return launch_status();
}

mlp_status launch_shadow(const float* w, void* wb, int wb_fmt, long long n,
                         const SgdSegments& segs, cudaStream_t st) {
  if (n <= 0) return MLP_OK;
  LaunchScope ls("shadow", st, n);
  launch_k(shadow_kernel, dim3(sgd_grid(n)), dim3(256), 0, st, w, static_cast<uint16_t*>(wb),
           wb_fmt, n, segs);
  return launch_status();
}

// ------------------------------------------------------------------ casts
// Inputs arrive as image bytes (value = byte / 255, IEEE division), fp32,
// bf16 or fp16; the tensor-core path wants bf16 or fp16, the SIMT path fp32.
// Source rows of `cols` values land in destination rows of pitch ld_dst.

__device__ __forceinline__ float load_in(const void* src, int src_dtype, size_t i) {
  if (src_dtype == MLP_DTYPE_U8) return (float)static_cast<const uint8_t*>(src)[i] / 255.0f;
  if (src_dtype == MLP_DTYPE_BF16 || src_dtype == MLP_DTYPE_F16)
    return f16bits_to_f32(static_cast<const uint16_t*>(src)[i], src_dtype);
  return static_cast<const float*>(src)[i];
}

// dst_dtype: MLP_DTYPE_F32, MLP_DTYPE_BF16 or MLP_DTYPE_F16.
// byte / 255 for a 16-bit destination: the product with fp32(1/255) rounds to
// the same bf16 and fp16 value as the IEEE quotient for every byte (checked
// exhaustively by the host tests), and costs one multiply instead of a divide.
__device__ __forceinline__ uint32_t bytes2_to_16(uint32_t w, int sh, int fmt) {
  const float r = 1.0f / 255.0f;
  return pack16x2_fmt((float)((w >> sh) & 0xffu) * r, (float)((w >> (sh + 8)) & 0xffu) * r, fmt);
}

__global__ void __launch_bounds__(256) cast_rows_kernel(const void* __restrict__ src,
                                                        int src_dtype, void* __restrict__ dst,
                                                        int dst_dtype, int rows, int cols,
                                                        int ld_dst) {
  pdl_wait();
  pdl_launch_dependents();
  const bool d16 = dst_dtype != MLP_DTYPE_F32;
  if (d16 && src_dtype == MLP_DTYPE_U8 && (cols & 15) == 0 && (ld_dst & 7) == 0) {
    // the whole matrix as 16-byte input chunks: 16 bytes in, 32 bytes out per
    // chunk, two chunks in flight per thread
    const int cpr = cols >> 4;
    const long long n = (long long)rows * cpr;
    const long long stride = (long long)gridDim.x * blockDim.x;
    const uint8_t* s8 = static_cast<const uint8_t*>(src);
    uint16_t* d16p = static_cast<uint16_t*>(dst);
    for (long long q0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; q0 < n;
         q0 += 2 * stride) {
      uint4 in[2];
      long long qq[2] = {q0, q0 + stride};
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (qq[k] < n) {
          const long long r = qq[k] / cpr, c = qq[k] - r * cpr;
          in[k] = __ldcs(reinterpret_cast<const uint4*>(s8 + r * cols) + c);
        }
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (qq[k] < n) {
          const long long r = qq[k] / cpr, c = qq[k] - r * cpr;
          const uint32_t* w = reinterpret_cast<const uint32_t*>(&in[k]);
          uint4 o0, o1;
          o0.x = bytes2_to_16(w[0], 0, dst_dtype);
          o0.y = bytes2_to_16(w[0], 16, dst_dtype);
          o0.z = bytes2_to_16(w[1], 0, dst_dtype);
          o0.w = bytes2_to_16(w[1], 16, dst_dtype);
          o1.x = bytes2_to_16(w[2], 0, dst_dtype);
          o1.y = bytes2_to_16(w[2], 16, dst_dtype);
          o1.z = bytes2_to_16(w[3], 0, dst_dtype);
          o1.w = bytes2_to_16(w[3], 16, dst_dtype);
          uint4* dq = reinterpret_cast<uint4*>(d16p + r * ld_dst) + 2 * c;
          dq[0] = o0;
          dq[1] = o1;
        }
    }
    return;
  }
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const size_t si = (size_t)r * cols, di = (size_t)r * ld_dst;
    if (d16 && src_dtype == MLP_DTYPE_U8 && (cols & 7) == 0 && (ld_dst & 7) == 0) {
      // 8 bytes in, 8 16-bit values (16 bytes) out per thread
      const uint2* s8 = reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(src) + si);
      uint4* dq = reinterpret_cast<uint4*>(static_cast<uint16_t*>(dst) + di);
      for (int q = threadIdx.x; q < cols / 8; q += blockDim.x) {
        const uint2 b = s8[q];
        uint4 o;
        o.x = bytes2_to_16(b.x, 0, dst_dtype);
        o.y = bytes2_to_16(b.x, 16, dst_dtype);
        o.z = bytes2_to_16(b.y, 0, dst_dtype);
        o.w = bytes2_to_16(b.y, 16, dst_dtype);
        dq[q] = o;
      }
    } else {
      for (int c = threadIdx.x; c < cols; c += blockDim.x) {
        const float v = load_in(src, src_dtype, si + c);
        if (d16) static_cast<uint16_t*>(dst)[di + c] = f32_to_16_fmt(v, dst_dtype);
        else static_cast<float*>(dst)[di + c] = v;
      }
    }
  }
}

mlp_status launch_cast_rows(const void* src, int src_dtype, void* dst, int dst_dtype, int rows,
                            int cols, int ld_dst, cudaStream_t st) {
  if (rows <= 0 || cols <= 0) return MLP_OK;
  // the vector path of the kernel needs 8-byte source rows and 16-byte
  // destination rows, which the row-size checks there and 16-byte base
  // pointers (checked by the callers) guarantee
  int blocks = rows < num_sms() * 16 ? rows : num_sms() * 16;
  if (dst_dtype != MLP_DTYPE_F32 && src_dtype == MLP_DTYPE_U8 && (cols & 15) == 0 &&
      (ld_dst & 7) == 0) {
    // flattened form: enough 256-thread blocks for two 16-byte chunks per
    // thread, at most 8 per SM
    const long long chunks = (long long)rows * (cols >> 4);
    const long long want = (chunks + 511) / 512;
    blocks = (int)(want < (long long)num_sms() * 8 ? want : (long long)num_sms() * 8);
    if (blocks < 1) blocks = 1;
  }
  LaunchScope ls("cast", st, (long long)rows * cols);
  launch_k(cast_rows_kernel, dim3(blocks), dim3(256), 0, st, src, src_dtype, dst, dst_dtype, rows,
           cols, ld_dst);
  return launch_status();
}

// ------------------------------------------------------------------ softmax xent
//
// "Capstone 5", "The minimum model" and "Read the worked reference": the loss
// kernel subtracts each row's maximum before exponentiating, so logits at
// +/-60 stay finite.  "The Work Moved Down a Layer", "The Debugging Lesson Was
// Numerical": the reductions run in fp32 with warp shuffles.
// One warp per row; lanes stride over the classes; the row max (with the
// lowest index among ties), the sum of exponentials and the loss are reduced
// with a fixed butterfly, so every lane holds identical values.

struct MaxIdx {
  float v;
  int i;
};

__device__ __forceinline__ MaxIdx warp_argmax(MaxIdx a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, a.v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, a.i, o);
    if (ov > a.v || (ov == a.v && oi < a.i)) { a.v = ov; a.i = oi; }
  }
  return a;
}

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

__device__ __forceinline__ float warp_max(float m) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

__device__ __forceinline__ float xent_row(const float* __restrict__ z, int label, int C,
                                          float inv_norm, void* dlog_row, int dl_dtype, int ldd,
                                          int* argmax_out, int lane) {
  label = label < 0 ? 0 : (label >= C ? C - 1 : label);  // keep the read in bounds
  MaxIdx best{-INFINITY, 0x7fffffff};
  for (int c = lane; c < C; c += 32) {
    const float v = z[c];
    if (v > best.v || (v == best.v && c < best.i)) { best.v = v; best.i = c; }
  }
  best = warp_argmax(best);
  const float m = best.v;
  float s = 0.f;
  for (int c = lane; c < C; c += 32) s += expf(z[c] - m);
  s = warp_sum(s);
  const float loss = m + logf(s) - z[label];
  if (dlog_row) {
    for (int c = lane; c < ldd; c += 32) {
      float d = 0.f;
      if (c < C) d = (expf(z[c] - m) / s - (c == label ? 1.f : 0.f)) * inv_norm;
      if (dl_dtype) static_cast<uint16_t*>(dlog_row)[c] = f32_to_16_fmt(d, dl_dtype);
      else static_cast<float*>(dlog_row)[c] = d;
    }
  }
  if (argmax_out && lane == 0) *argmax_out = best.i;
  return loss;
}

// Two fp32 values in one 64-bit register for the paired fp32 instructions of
// sm_100 and later (two independent round-to-nearest operations each).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// The hardware base-2 exponential (PTX ex2.approx, results below 2^-126
// flushed to zero).
__device__ __forceinline__ float ex2_hw(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Rows of up to 1024 classes whose logits start on 16-byte boundaries: one
// warp holds the row in registers (4 values per lane per 128-class segment,
// classes past C as -inf), keeps their exponentials there and writes dZ from
// them.  zy is the label's logit.
template <int NSEG>
__device__ __forceinline__ float xent_row_regs(float (&v)[NSEG][4], float zy, int label, int C,
                                               float inv_norm, void* dlog_row, int dl_dtype,
                                               int ldd, int* argmax_out, int lane) {
  // the row maximum; its first index only when the caller asks for it
  float m;
  int best_i = 0;
  if (argmax_out) {
    MaxIdx best{-INFINITY, 0x7fffffff};
#pragma unroll
    for (int g = 0; g < NSEG; ++g) {
      const int c0 = g * 128 + lane * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (v[g][e] > best.v || (v[g][e] == best.v && c0 + e < best.i)) {
          best.v = v[g][e];
          best.i = c0 + e;
        }
    }
    best = warp_argmax(best);
    m = best.v;
    best_i = best.i;
  } else {
    m = -INFINITY;
#pragma unroll
    for (int g = 0; g < NSEG; ++g)
#pragma unroll
      for (int e = 0; e < 4; ++e) m = fmaxf(m, v[g][e]);
    m = warp_max(m);
  }
  // e^(z - m) as 2^(z log2(e) - m log2(e)): the argument as one fused
  // multiply-add per element (two per paired instruction), whose roundings
  // (of m log2(e) and of the result) shift it by about |m| 2^-23, a relative
  // error near 1e-6 of each exponential, common to the row for the m part;
  // well inside the fp32 dZ and loss tolerances.  Classes past C hold -inf,
  // whose exponential is 0.  The row sum runs in two interleaved halves.
  constexpr float kLog2e = 1.4426950408889634f;
  const uint64_t l2 = f2_pack(kLog2e, kLog2e);
  const uint64_t ml2 = f2_pack(-m * kLog2e, -m * kLog2e);
  uint64_t s2 = f2_pack(0.f, 0.f);
#pragma unroll
  for (int g = 0; g < NSEG; ++g)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float t0, t1;
      f2_unpack(f2_fma(f2_pack(v[g][2 * h], v[g][2 * h + 1]), l2, ml2), t0, t1);
      v[g][2 * h] = ex2_hw(t0);
      v[g][2 * h + 1] = ex2_hw(t1);
      s2 = f2_add(s2, f2_pack(v[g][2 * h], v[g][2 * h + 1]));
    }
  float s_lo, s_hi;
  f2_unpack(s2, s_lo, s_hi);
  const float s = warp_sum(s_lo + s_hi);
  const float loss = m + logf(s) - zy;
  if (dlog_row) {
    // dZ = (softmax - onehot) / B: exp(z - m) times the row's one factor
    // 1 / (s B) (zero past C, where the exponentials are zero), and 1 / B off
    // the label's entry in the lane and segment that hold it
    const float a = inv_norm / s;
    const uint64_t a2 = f2_pack(a, a);
    const int lab_lane = (label & 127) >> 2, lab_seg = label >> 7, lab_e = label & 3;
#pragma unroll
    for (int g = 0; g < NSEG; ++g) {
      const int c0 = g * 128 + lane * 4;
      float d[4];
      f2_unpack(f2_mul(f2_pack(v[g][0], v[g][1]), a2), d[0], d[1]);
      f2_unpack(f2_mul(f2_pack(v[g][2], v[g][3]), a2), d[2], d[3]);
      if (g == lab_seg && lane == lab_lane) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (e == lab_e) d[e] -= inv_norm;
      }
      if (c0 + 3 < ldd) {
        if (dl_dtype) {
          uint2 o;
          o.x = pack16x2_fmt(d[0], d[1], dl_dtype);
          o.y = pack16x2_fmt(d[2], d[3], dl_dtype);
          *reinterpret_cast<uint2*>(static_cast<uint16_t*>(dlog_row) + c0) = o;
        } else {
          *reinterpret_cast<float4*>(static_cast<float*>(dlog_row) + c0) =
              make_float4(d[0], d[1], d[2], d[3]);
        }
      } else {
        for (int e = 0; e < 4 && c0 + e < ldd; ++e) {
          if (dl_dtype) static_cast<uint16_t*>(dlog_row)[c0 + e] = f32_to_16_fmt(d[e], dl_dtype);
          else static_cast<float*>(dlog_row)[c0 + e] = d[e];
        }
      }
    }
    // padding columns beyond the last 128-class segment
    for (int c = NSEG * 128 + lane; c < ldd; c += 32) {
      if (dl_dtype) static_cast<uint16_t*>(dlog_row)[c] = 0;
      else static_cast<float*>(dlog_row)[c] = 0.f;
    }
  }
  if (argmax_out && lane == 0) *argmax_out = best_i;
  return loss;
}

// Warp w of block b takes rows b * 8 + w, then every 8 * gridDim.x-th row
// after it (two blocks per SM) and adds their losses in that order;
// partial[b] is the block's sum.  Each warp keeps its next kXentDepth rows in
// flight: bulk copies into its own shared-memory row buffers, completing on
// one mbarrier per buffer, issued as soon as the buffer's row has been read
// into registers.  The labels of those rows are loaded as the copies are
// issued.  Waits are bounded; a warp that gives up records the timeout and
// waits (bounded again) for its copies still in flight before the block exits.
constexpr int kXentDepth = 3;

template <int NSEG>
constexpr size_t xent_rows_smem() {
  return (size_t)8 * kXentDepth * NSEG * 128 * sizeof(float);
}

template <int NSEG>
__global__ void __launch_bounds__(256, 2) xent_rows_regs_kernel(
    const float* __restrict__ logits, int ldl, const int* __restrict__ labels, int B, int C,
    float* __restrict__ partial, void* dlog, int dl_dtype, int ldd, int* argmax,
    unsigned long long wait_ns, int* err) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int ROWF = NSEG * 128;
  extern __shared__ __align__(128) float xent_rows[];
  __shared__ __align__(8) uint64_t bars[8][kXentDepth];
  __shared__ float part[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* buf = xent_rows + warp * kXentDepth * ROWF;
  const int stride = gridDim.x * 8;
  const int first = blockIdx.x * 8 + warp;
  const uint32_t bytes = ((uint32_t)C * 4u + 15u) & ~15u;  // within the row pitch (ldl % 4 == 0)
  const int c_pad = (C + 3) & ~3;  // classes [C, c_pad) arrive with the row and are masked
  if (lane == 0) {
    for (int d = 0; d < kXentDepth; ++d) ptx::mbar_init(&bars[warp][d], 1);
    ptx::fence_mbar_init();
  }
  // the buffers' classes past the copied bytes hold -inf for the whole launch
  for (int d = 0; d < kXentDepth; ++d)
    for (int c = c_pad + lane; c < ROWF; c += 32) buf[d * ROWF + c] = -INFINITY;
  __syncwarp();
  // the first rows of this warp, and their labels
  int lab[kXentDepth];
#pragma unroll
  for (int d = 0; d < kXentDepth; ++d) {
    const int r = first + d * stride;
    lab[d] = r < B ? labels[r] : 0;
    if (lane == 0 && r < B) {
      ptx::mbar_arrive_expect_tx(&bars[warp][d], bytes);
      ptx::bulk_load_global(buf + d * ROWF, logits + (size_t)r * ldl, bytes, &bars[warp][d]);
    }
  }
  float li = 0.f;
  int k = 0;
  bool ok = true;
  for (int r = first; r < B; r += stride, ++k) {
    const int d = k % kXentDepth;
    if (!ptx::mbar_wait_bounded(&bars[warp][d], (uint32_t)((k / kXentDepth) & 1), wait_ns, err,
                                DEVERR_TIMEOUT_PRODUCER)) {
      ok = false;
      break;
    }
    float* row = buf + d * ROWF;
    if (c_pad != C) {  // the copied row's padding past C
      if (lane < c_pad - C) row[C + lane] = -INFINITY;
      __syncwarp();
    }
    float v[NSEG][4];
#pragma unroll
    for (int g = 0; g < NSEG; ++g) {
      const float4 q = *reinterpret_cast<const float4*>(row + g * 128 + lane * 4);
      v[g][0] = q.x; v[g][1] = q.y; v[g][2] = q.z; v[g][3] = q.w;
    }
    const int label = lab[0] < 0 ? 0 : (lab[0] >= C ? C - 1 : lab[0]);
    const float zy = row[label];
#pragma unroll
    for (int j = 0; j + 1 < kXentDepth; ++j) lab[j] = lab[j + 1];
    // every lane has read the buffer: refill it with the row kXentDepth ahead
    __syncwarp();
    const int rn = r + kXentDepth * stride;
    lab[kXentDepth - 1] = rn < B ? labels[rn] : 0;
    if (lane == 0 && rn < B) {
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive_expect_tx(&bars[warp][d], bytes);
      ptx::bulk_load_global(buf + d * ROWF, logits + (size_t)rn * ldl, bytes, &bars[warp][d]);
    }
    void* drow = nullptr;
    if (dlog) drow = dl_dtype ? (void*)(static_cast<uint16_t*>(dlog) + (size_t)r * ldd)
                             : (void*)(static_cast<float*>(dlog) + (size_t)r * ldd);
    li += xent_row_regs<NSEG>(v, zy, label, C, 1.0f / (float)B, drow, dl_dtype, ldd,
                              argmax ? argmax + r : nullptr, lane);
  }
  if (!ok && lane == 0) {
    // copies issued and not yet consumed: rows k, k + 1, ... of this warp
    for (int j = k; j < k + kXentDepth && first + j * stride < B; ++j)
      ptx::mbar_wait_bounded(&bars[warp][j % kXentDepth], (uint32_t)((j / kXentDepth) & 1),
                             wait_ns, err, DEVERR_TIMEOUT_TEARDOWN);
  }
  if (lane == 0) part[warp] = li;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += part[w];
    partial[blockIdx.x] = t;
  }
}

// Small batches: one block, 8 warps striding over the rows; the block also
// forms the mean (warp w sums its rows in order, then warp sums in order).
__global__ void __launch_bounds__(256) xent_single_block_kernel(
    const float* __restrict__ logits, int ldl, const int* __restrict__ labels, int B, int C,
    float* __restrict__ loss_out, void* dlog, int dl_dtype, int ldd, int* argmax, int* err) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float part[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float inv_norm = 1.0f / (float)B;
  float acc = 0.f;
  for (int r = warp; r < B; r += 8) {
    void* drow = nullptr;
    if (dlog) drow = dl_dtype ? (void*)(static_cast<uint16_t*>(dlog) + (size_t)r * ldd)
                             : (void*)(static_cast<float*>(dlog) + (size_t)r * ldd);
    acc += xent_row(logits + (size_t)r * ldl, labels[r], C, inv_norm, drow, dl_dtype, ldd,
                    argmax ? argmax + r : nullptr, lane);
  }
  if (lane == 0) part[warp] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += part[w];
    const float loss = t / (float)B;
    check_loss_finite(loss, err);
    if (loss_out) *loss_out = loss;
  }
}

// Small heads (C <= 32) of small batches (B <= 512): one row per thread of
// a single block, so every row's max, sum and dZ come out of one pass with
// one round trip to memory (the row routine of xent_row.cuh, shared with the
// loss epilogue of the logits GEMM); the batch mean is a fixed-order tree sum.
template <int NC>
__device__ __forceinline__ float xent_lane_row(const float* __restrict__ z_row, int label, int C,
                                               float inv, void* dlog_row, int dl_dtype, int ldd,
                                               int* argmax) {
  float z[NC], d[NC];
#pragma unroll
  for (int j = 0; j < NC; ++j) z[j] = j < C ? z_row[j] : 0.f;
  int am;
  const float li = xent_row_small<NC>(z, C, label, inv, d, am);
  if (dlog_row) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < ldd) {
        const float v = j < NC ? d[j % NC] : 0.f;
        if (dl_dtype) static_cast<uint16_t*>(dlog_row)[j] = f32_to_16_fmt(v, dl_dtype);
        else static_cast<float*>(dlog_row)[j] = v;
      }
    }
  }
  if (argmax) *argmax = am;
  return li;
}

__global__ void __launch_bounds__(512) xent_lane_rows_kernel(
    const float* __restrict__ logits, int ldl, const int* __restrict__ labels, int B, int C,
    float* __restrict__ loss_out, void* dlog, int dl_dtype, int ldd, int* argmax, int* err) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[512];
  const int r = threadIdx.x;
  float li = 0.f;
  if (r < B) {
    const float inv = 1.0f / (float)B;
    void* drow = nullptr;
    if (dlog) drow = dl_dtype ? (void*)(static_cast<uint16_t*>(dlog) + (size_t)r * ldd)
                             : (void*)(static_cast<float*>(dlog) + (size_t)r * ldd);
    int* am = argmax ? argmax + r : nullptr;
    li = C <= 16 ? xent_lane_row<16>(logits + (size_t)r * ldl, labels[r], C, inv, drow, dl_dtype,
                                     ldd, am)
                 : xent_lane_row<32>(logits + (size_t)r * ldl, labels[r], C, inv, drow, dl_dtype,
                                     ldd, am);
  }
  red[r] = li;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (r < w) red[r] += red[r + w];
    __syncthreads();
  }
  if (r == 0) {
    const float loss = red[0] / (float)B;
    check_loss_finite(loss, err);
    if (loss_out) *loss_out = loss;
  }
}

// Large batches: one row per warp, one partial per block, then a one-block
// fixed-order sum.
__global__ void __launch_bounds__(256) xent_rows_kernel(
    const float* __restrict__ logits, int ldl, const int* __restrict__ labels, int B, int C,
    float* __restrict__ partial, void* dlog, int dl_dtype, int ldd, int* argmax) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float part[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + warp;
  float li = 0.f;
  if (r < B) {
    void* drow = nullptr;
    if (dlog) drow = dl_dtype ? (void*)(static_cast<uint16_t*>(dlog) + (size_t)r * ldd)
                             : (void*)(static_cast<float*>(dlog) + (size_t)r * ldd);
    li = xent_row(logits + (size_t)r * ldl, labels[r], C, 1.0f / (float)B, drow, dl_dtype, ldd,
                  argmax ? argmax + r : nullptr, lane);
  }
  if (lane == 0) part[warp] = li;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += part[w];
    partial[blockIdx.x] = t;
  }
}

// Sum of `n` partials in a fixed order, times `scale`, into *out.
// out = (sum of the n partials in a fixed order) / divisor: the mean of a
// loss, so a non-finite result is recorded in the device error word.
__global__ void __launch_bounds__(256) sum_partials_kernel(const float* __restrict__ partial,
                                                           long long n, float divisor,
                                                           float* __restrict__ out, int* err) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[256];
  float t = 0.f;
  for (long long i = threadIdx.x; i < n; i += 256) t += partial[i];
  red[threadIdx.x] = t;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const float loss = red[0] / divisor;
    check_loss_finite(loss, err);
    *out = loss;
  }
}

size_t xent_workspace_bytes(int B) {
  if (B <= 256) return 0;
  return (size_t)((B + 7) / 8) * sizeof(float);
}

mlp_status launch_xent(const float* logits, int ldl, const int* labels, int B, int C,
                       float* loss_out, void* dlog, int dl_dtype, int ldd, int* argmax,
                       void* ws, cudaStream_t st) {
  if (B <= 0) return MLP_OK;
  if (C <= 32 && ldd <= 32 && B <= 512) {
    int threads = 32;
    while (threads < B) threads *= 2;  // a power of two for the tree sum
    LaunchScope ls("xent", st, B, C);
    launch_k(xent_lane_rows_kernel, dim3(1), dim3(threads), 0, st, logits, ldl, labels, B, C,
             loss_out, dlog, dl_dtype, ldd, argmax, device_error_word());
    return launch_status();
  }
  if (B <= 256) {
    LaunchScope ls("xent", st, B, C);
    launch_k(xent_single_block_kernel, dim3(1), dim3(256), 0, st, logits, ldl, labels, B, C,
             loss_out, dlog, dl_dtype, ldd, argmax, device_error_word());
    return launch_status();
  }
  int blocks = (B + 7) / 8;
  float* partial = static_cast<float*>(ws);
  const bool vec = C <= 1024 && (ldl % 4) == 0 && aligned16(logits) &&
                   (!dlog || ((ldd % 4) == 0 && aligned16(dlog)));
  // the register-resident rows kernel loops over rows: one wave of blocks
  // (at most as many partials as the workspace holds, one per 8 rows)
  if (vec && blocks > num_sms() * 2) blocks = num_sms() * 2;
  {
  LaunchScope ls("xent", st, B, C);
  static bool configured = false;
  if (vec && !configured) {
    if (cudaFuncSetAttribute(xent_rows_regs_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)xent_rows_smem<2>()) != cudaSuccess ||
        cudaFuncSetAttribute(xent_rows_regs_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)xent_rows_smem<8>()) != cudaSuccess)
      return MLP_ERR_CUDA;
    configured = true;
  }
  const unsigned long long wait_ns = wait_limit_ns();
  if (vec && C <= 256)
    launch_k(xent_rows_regs_kernel<2>, dim3(blocks), dim3(256), xent_rows_smem<2>(), st, logits,
             ldl, labels, B, C, partial, dlog, dl_dtype, ldd, argmax, wait_ns,
             device_error_word());
  else if (vec)
    launch_k(xent_rows_regs_kernel<8>, dim3(blocks), dim3(256), xent_rows_smem<8>(), st, logits,
             ldl, labels, B, C, partial, dlog, dl_dtype, ldd, argmax, wait_ns,
             device_error_word());
  else
    launch_k(xent_rows_kernel, dim3(blocks), dim3(256), 0, st, logits, ldl, labels, B, C, partial, dlog, dl_dtype,
                                             ldd, argmax);
  }
  MLP_CHECK(launch_status());
  if (loss_out) {
    LaunchScope ls("sum_partials", st, blocks);
    launch_k(sum_partials_kernel, dim3(1), dim3(256), 0, st, partial, blocks, (float)B, loss_out,
             device_error_word());
    return launch_status();
  }
  return MLP_OK;
}

// ------------------------------------------------------------------ column sums
//
// "Capstone 5", "Check your mapping": each bias gradient is a column
// reduction across the batch.  Pass 1: block (32 x 8 threads) covers 64
// columns of one row chunk, each thread two adjacent columns (a warp reads 64
// consecutive elements of a row); the 8 row-strided partial sums are added in
// order.  Pass 2 (only when there is more than one chunk) adds the chunk
// partials in order.

template <typename T>
__device__ __forceinline__ float ldf(const T* p);
template <>
__device__ __forceinline__ float ldf<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
  return bf16_to_f32(*p);
}
template <>
__device__ __forceinline__ float ldf<__half>(const __half* p) {
  return __half2float(*p);
}

template <typename T>
__global__ void __launch_bounds__(256) colsum_pass1_kernel(const T* __restrict__ X, int rows,
                                                           int cols, int ld, int rows_per_chunk,
                                                           float* __restrict__ dst) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float s[8][65];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int c = blockIdx.x * 64 + 2 * tx;
  const int r0 = blockIdx.y * rows_per_chunk;
  const int r1 = min(rows, r0 + rows_per_chunk);
  float a0 = 0.f, a1 = 0.f;
  for (int r = r0 + ty; r < r1; r += 8) {
    const T* row = X + (size_t)r * ld;
    if (c < cols) a0 += ldf(row + c);
    if (c + 1 < cols) a1 += ldf(row + c + 1);
  }
  s[ty][2 * tx] = a0;
  s[ty][2 * tx + 1] = a1;
  __syncthreads();
  if (ty == 0) {
    for (int e = 0; e < 2; ++e) {
      const int cc = c + e;
      if (cc < cols) {
        float t = 0.f;
        for (int k = 0; k < 8; ++k) t += s[k][2 * tx + e];
        dst[(size_t)blockIdx.y * cols + cc] = t;
      }
    }
  }
}

// Vector form: each lane reads 16 bytes of a row (8 bf16 / fp16 or 4 fp32 columns),
// a warp covers 512 contiguous bytes, 8 warps stride over the rows of the
// chunk (4 rows in flight per lane), then the warps' sums are added in order.
template <typename T>
__global__ void __launch_bounds__(256) colsum_vec_kernel(const T* __restrict__ X, int rows,
                                                         int cols, int ld, int rows_per_chunk,
                                                         float* __restrict__ dst) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int V = 16 / sizeof(T);          // columns per lane
  constexpr int BC = 32 * V;                 // columns per block
  __shared__ float s[8][BC + 1];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c0 = blockIdx.x * BC + lane * V;
  const int r0 = blockIdx.y * rows_per_chunk;
  const int r1 = min(rows, r0 + rows_per_chunk);
  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  if (c0 < cols) {
    int r = r0 + w;
    for (; r + 24 < r1; r += 32) {
      uint4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) q[u] = __ldcs(reinterpret_cast<const uint4*>(X + (size_t)(r + 8 * u) * ld + c0));
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const T* t = reinterpret_cast<const T*>(&q[u]);
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] += ldf(t + e);
      }
    }
    for (; r < r1; r += 8) {
      const uint4 q = __ldcs(reinterpret_cast<const uint4*>(X + (size_t)r * ld + c0));
      const T* t = reinterpret_cast<const T*>(&q);
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] += ldf(t + e);
    }
  }
#pragma unroll
  for (int e = 0; e < V; ++e) s[w][lane * V + e] = acc[e];
  __syncthreads();
  for (int c = threadIdx.x; c < BC; c += 256) {
    const int cc = blockIdx.x * BC + c;
    if (cc < cols) {
      float t = 0.f;
      for (int k = 0; k < 8; ++k) t += s[k][c];
      dst[(size_t)blockIdx.y * cols + cc] = t;
    }
  }
}

__global__ void colsum_pass2_kernel(const float* __restrict__ partial, int chunks, int cols,
                                    float* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  float t = 0.f;
  for (int k = 0; k < chunks; ++k) t += partial[(size_t)k * cols + c];
  out[c] = t;
}

// Linear-order form (MLP_ORDER_LINEAR): thread c adds rows 0, 1, ..., rows-1
// of column c into one fp32 accumulator, the plain loop a CPU would run; the
// warp's 32 columns are read together, so each row step is one coalesced
// load per warp.
template <typename T>
__global__ void __launch_bounds__(128) colsum_linear_kernel(const T* __restrict__ X, int rows,
                                                            int cols, int ld,
                                                            float* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  float s = 0.f;
  for (int r = 0; r < rows; ++r) s += ldf(X + (size_t)r * ld + c);
  out[c] = s;
}

void colsum_plan(int rows, int cols, int* chunks, int* rows_per_chunk) {
  (void)cols;
  int ch = (rows + 511) / 512;
  if (ch > 32) ch = 32;
  if (ch < 1) ch = 1;
  int rpc = (rows + ch - 1) / ch;
  rpc = (rpc + 7) / 8 * 8;
  ch = rpc > 0 ? (rows + rpc - 1) / rpc : 1;
  if (ch < 1) ch = 1;
  *chunks = ch;
  *rows_per_chunk = rpc > 0 ? rpc : 8;
}

size_t colsum_workspace_bytes(int rows, int cols) {
  int ch, rpc;
  colsum_plan(rows, cols, &ch, &rpc);
  return ch > 1 ? (size_t)ch * cols * sizeof(float) : 0;
}

// dtype: MLP_DTYPE_F32, MLP_DTYPE_BF16 or MLP_DTYPE_F16.
template <typename T>
void launch_colsum_t(const T* X, int rows, int cols, int ld, int ch, int rpc, float* dst,
                     bool vec, cudaStream_t st) {
  LaunchScope ls("colsum", st, rows, cols);
  if (vec) {
    constexpr int bc = 32 * (16 / (int)sizeof(T));
    dim3 g((cols + bc - 1) / bc, ch);
    launch_k(colsum_vec_kernel<T>, g, dim3(256), 0, st, X, rows, cols, ld, rpc, dst);
  } else {
    dim3 grid((cols + 63) / 64, ch);
    launch_k(colsum_pass1_kernel<T>, grid, dim3(256), 0, st, X, rows, cols, ld, rpc, dst);
  }
}

mlp_status launch_colsum(const void* X, int dtype, int rows, int cols, int ld, float* out,
                         void* ws, cudaStream_t st) {
  if (cols <= 0) return MLP_OK;
  if (linear_order()) {
    LaunchScope ls("colsum_linear", st, rows, cols);
    const dim3 g((cols + 127) / 128);
    if (dtype == MLP_DTYPE_BF16)
      launch_k(colsum_linear_kernel<__nv_bfloat16>, g, dim3(128), 0, st,
               static_cast<const __nv_bfloat16*>(X), rows, cols, ld, out);
    else if (dtype == MLP_DTYPE_F16)
      launch_k(colsum_linear_kernel<__half>, g, dim3(128), 0, st, static_cast<const __half*>(X),
               rows, cols, ld, out);
    else
      launch_k(colsum_linear_kernel<float>, g, dim3(128), 0, st, static_cast<const float*>(X),
               rows, cols, ld, out);
    return launch_status();
  }
  int ch, rpc;
  colsum_plan(rows, cols, &ch, &rpc);
  float* dst = ch > 1 ? static_cast<float*>(ws) : out;
  const bool h16 = dtype != MLP_DTYPE_F32;
  const bool vec = aligned16(X) && (h16 ? (cols % 8 == 0 && ld % 8 == 0)
                                        : (cols % 4 == 0 && ld % 4 == 0));
  if (dtype == MLP_DTYPE_BF16)
    launch_colsum_t(static_cast<const __nv_bfloat16*>(X), rows, cols, ld, ch, rpc, dst, vec, st);
  else if (dtype == MLP_DTYPE_F16)
    launch_colsum_t(static_cast<const __half*>(X), rows, cols, ld, ch, rpc, dst, vec, st);
  else
    launch_colsum_t(static_cast<const float*>(X), rows, cols, ld, ch, rpc, dst, vec, st);
  MLP_CHECK(launch_status());
  if (ch > 1) {
    LaunchScope ls("colsum_final", st, ch, cols);
    launch_k(colsum_pass2_kernel, dim3((cols + 255) / 256), dim3(256), 0, st, dst, ch, cols, out);
    return launch_status();
  }
  return MLP_OK;
}

// ------------------------------------------------------------------ MSE
// loss = mean((y - t)^2), dy = 2 (y - t) / n; y, t, dy bf16.  Each thread
// handles 8 consecutive elements per 16-byte load; block partials are summed
// in a fixed order by sum_partials_kernel.

__global__ void __launch_bounds__(256) mse_kernel(const __nv_bfloat16* __restrict__ y,
                                                  const __nv_bfloat16* __restrict__ t,
                                                  long long n, __nv_bfloat16* __restrict__ dy,
                                                  float* __restrict__ partial) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[256];
  const float scale = 2.0f / (float)n;
  const long long n8 = n >> 3;
  const long long stride = (long long)gridDim.x * blockDim.x;
  float acc = 0.f;
  for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < n8; q += stride) {
    const uint4 yv = __ldcs(reinterpret_cast<const uint4*>(y) + q);
    const uint4 tv = __ldcs(reinterpret_cast<const uint4*>(t) + q);
    const __nv_bfloat162* yp = reinterpret_cast<const __nv_bfloat162*>(&yv);
    const __nv_bfloat162* tp = reinterpret_cast<const __nv_bfloat162*>(&tv);
    uint4 out;
    uint32_t* op = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 a = __bfloat1622float2(yp[e]);
      const float2 b = __bfloat1622float2(tp[e]);
      const float d0 = a.x - b.x, d1 = a.y - b.y;
      acc += d0 * d0;
      acc += d1 * d1;
      op[e] = pack_bf16x2(d0 * scale, d1 * scale);
    }
    if (dy) __stcs(reinterpret_cast<uint4*>(dy) + q, out);
  }
  if (blockIdx.x == 0) {
    for (long long i = (n8 << 3) + threadIdx.x; i < n; i += blockDim.x) {
      const float d = bf16_to_f32(y[i]) - bf16_to_f32(t[i]);
      acc += d * d;
      if (dy) dy[i] = f32_to_bf16(d * scale);
    }
  }
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) partial[blockIdx.x] = red[0];
}

int mse_blocks(long long n) {
  long long q = (n / 8 + 255) / 256;
  const long long cap = 1024;  // fixed cap: the partition depends only on n
  if (q > cap) q = cap;
  if (q < 1) q = 1;
  return (int)q;
}

size_t mse_ws_bytes(long long n) { return (size_t)mse_blocks(n) * sizeof(float); }

mlp_status launch_mse(const void* y, const void* t, long long n, float* loss_out, void* dy,
                      void* ws, cudaStream_t st) {
  if (n <= 0) return MLP_OK;
  const int blocks = mse_blocks(n);
  float* partial = static_cast<float*>(ws);
  {
  LaunchScope ls("mse", st, n);
  launch_k(mse_kernel, dim3(blocks), dim3(256), 0, st, static_cast<const __nv_bfloat16*>(y),
                                     static_cast<const __nv_bfloat16*>(t), n,
                                     static_cast<__nv_bfloat16*>(dy), partial);
  }
  MLP_CHECK(launch_status());
  if (loss_out) {
    LaunchScope ls("sum_partials", st, blocks);
    launch_k(sum_partials_kernel, dim3(1), dim3(256), 0, st, partial, blocks, (float)n, loss_out,
             device_error_word());
    return launch_status();
  }
  return MLP_OK;
}

// ------------------------------------------------------------------ row RMS
// r = 1 / sqrt(ss / d + eps) per token, ss its squares summed per lane in
// index order (16-byte loads of 8 bf16) and across the lanes by a fixed
// butterfly ("Full-Depth MLP Megakernel + Fused Attention Preprocessing",
// "What Worked": the RMSNorm in front of the QKV projection, gain 1, folded
// into the projection's epilogue as this per-token scale).  A warp takes 4
// consecutive tokens and requests the first 2 x 32 chunks of all four rows
// (rows of up to 512 values whole) before summing any: 4 KiB in flight per
// warp.  The loads leave the rows in L2 for the projection that reads them
// next.
constexpr int kRstdTok = 4, kRstdAhead = 2;

__global__ void __launch_bounds__(256) row_rstd_kernel(const __nv_bfloat16* __restrict__ x,
                                                       long long T, int d, float eps,
                                                       float* __restrict__ rstd) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long t0 = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * kRstdTok;
  if (t0 >= T) return;
  const int chunks = d / 8;
  uint4 v[kRstdTok][kRstdAhead];
#pragma unroll
  for (int j = 0; j < kRstdTok; ++j) {
    const uint4* row = reinterpret_cast<const uint4*>(x + (t0 + j) * d);
#pragma unroll
    for (int i = 0; i < kRstdAhead; ++i)
      v[j][i] = t0 + j < T && lane + 32 * i < chunks ? __ldg(row + lane + 32 * i)
                                                     : make_uint4(0u, 0u, 0u, 0u);
  }
  float ss[kRstdTok];
#pragma unroll
  for (int j = 0; j < kRstdTok; ++j) {
    ss[j] = 0.f;
    auto add = [&](const uint4& c) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&c);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        ss[j] = fmaf(f.x, f.x, ss[j]);
        ss[j] = fmaf(f.y, f.y, ss[j]);
      }
    };
#pragma unroll
    for (int i = 0; i < kRstdAhead; ++i) add(v[j][i]);
    if (t0 + j < T) {
      const uint4* row = reinterpret_cast<const uint4*>(x + (t0 + j) * d);
      for (int q = lane + 32 * kRstdAhead; q < chunks; q += 32) add(__ldg(row + q));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int j = 0; j < kRstdTok; ++j) ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], o);
  if (lane < kRstdTok && t0 + lane < T) {
    float s = ss[0];
#pragma unroll
    for (int j = 1; j < kRstdTok; ++j)
      if (lane == j) s = ss[j];
    rstd[t0 + lane] = 1.0f / sqrtf(s / (float)d + eps);
  }
}

mlp_status launch_row_rstd(const void* x, long long T, int d, float eps, float* rstd,
                           cudaStream_t st) {
  if (T <= 0) return MLP_OK;
  LaunchScope ls("row_rstd", st, T, d);
  launch_k(row_rstd_kernel, dim3((unsigned)((T + 8 * kRstdTok - 1) / (8 * kRstdTok))), dim3(256),
           0, st, static_cast<const __nv_bfloat16*>(x), T, d, eps, rstd);
  return launch_status();
}

// ------------------------------------------------------------------ ones columns

// dtype: MLP_DTYPE_F32, MLP_DTYPE_BF16 or MLP_DTYPE_F16.
__global__ void ones_cols_kernel(OnesCols oc, int rows, int dtype) {
  pdl_wait();
  pdl_launch_dependents();
  const int k = blockIdx.y;
  const int col = oc.col[k], ld = oc.ld[k];
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x) {
    for (int c = col; c < ld; ++c) {
      const float v = c == col ? 1.f : 0.f;
      if (dtype != MLP_DTYPE_F32)
        static_cast<uint16_t*>(oc.ptr[k])[(size_t)r * ld + c] = f32_to_16_fmt(v, dtype);
      else static_cast<float*>(oc.ptr[k])[(size_t)r * ld + c] = v;
    }
  }
}

mlp_status launch_ones_cols(const OnesCols& oc, int rows, int dtype, cudaStream_t st) {
  if (oc.n <= 0 || rows <= 0) return MLP_OK;
  LaunchScope ls("ones_cols", st, rows, oc.n);
  dim3 grid((rows + 255) / 256, oc.n);
  launch_k(ones_cols_kernel, dim3(grid), dim3(256), 0, st, oc, rows, dtype);
  return launch_status();
}

// ------------------------------------------------------------------ wait self-test
// One thread waits on a barrier that nothing arrives at; the bounded wait
// gives up after limit_ns, records the timeout and the kernel returns.

__global__ void wait_selftest_kernel(unsigned long long limit_ns, int* err) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    ptx::mbar_wait_bounded(&bar, 0, limit_ns, err, DEVERR_TIMEOUT_PEER);
  }
}

mlp_status launch_wait_selftest(unsigned long long limit_ns, cudaStream_t st) {
  int* err = device_error_word();
  if (!err) return MLP_ERR_CUDA;
  LaunchScope ls("wait_selftest", st);
  launch_k(wait_selftest_kernel, dim3(1), dim3(32), 0, st, limit_ns, err);
  return launch_status();
}

}  // namespace mlp
