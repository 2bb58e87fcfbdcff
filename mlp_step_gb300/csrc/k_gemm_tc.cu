// tcgen05 GEMM for sm_103a: bf16 operands fed by TMA into 128-byte-swizzled
// shared-memory stages, fp32 accumulation in tensor memory, fp32 epilogue
// (bias, ReLU, ReLU-mask) and a bf16 or fp32 store.
//
// "The Work Moved Down a Layer", "The Debugging Lesson Was Numerical": low
// precision only for the matrix inputs; the accumulator stays fp32 and bias
// and activation are applied in fp32 before the final conversion.  "Capstone 5:
// train a network with your CUDA kernels", "Read the worked reference": bias
// and ReLU in the epilogue; "Work through the backward pass": dW = X^T dH and
// dX = dH W^T read an operand transposed -- here the transposition is the
// operand's major-ness in the MMA descriptors (MN-major tiles), so no copy is
// ever made.  "Tile the data": operand tiles are reused from shared memory by
// a 128 x BN output tile.
//
// Structure: persistent kernel, one CTA per SM, 6 warps:
//   warp 0    TMA producer (one lane): fills a STAGES-deep ring of A/B tiles;
//   warp 1    tensor-memory owner and MMA issuer (one lane): 4 x (128 x BN x 16)
//             MMAs per 64-wide k-block, commits each stage back to the
//             producer and each finished tile to the epilogue;
//   warps 2-5 epilogue: tcgen05.ld of their 32-lane quarter of the
//             accumulator, fp32 epilogue, vector stores.
// Two accumulators (2 x BN tensor-memory columns) let the epilogue of tile i
// overlap the MMAs of tile i+1.  Every mbarrier wait is bounded; a timeout is
// recorded in the device error word and the CTA winds down cleanly.
#include <cstdlib>
#include <cstring>

#include "kernels.cuh"
#include "ptx.cuh"
#include "trace.cuh"
#include "xent_row.cuh"

namespace mlp {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 192;

struct TcParams {
  int M, N, K;
  int a_mn, b_mn;
  int tiles_m, tiles_n, num_tiles, k_blocks;
  const float* bias;
  int act;
  const __nv_bfloat16* mask;
  int ldm;
  void* C;
  int ldc;
  int c_bf16;  // C is 16-bit (bf16, or fp16 when f16 is set)
  int f16;     // operands and 16-bit outputs are fp16 rather than bf16
  unsigned long long wait_ns;
  int* err;
  // split-K: each work unit covers k-blocks [s*kb_per_split, (s+1)*kb_per_split)
  // of one tile and stores raw fp32 sums into partial[s][M][ldp]
  int splits, kb_per_split, ldp;
  float* partial;
  // fused softmax cross entropy (single tile) and momentum SGD epilogues
  const int* xent_labels;
  __nv_bfloat16* xent_dlog;
  int xent_ldd;
  float* xent_loss;
  int* xent_argmax;
  int xent_norm;
  float* sgd_w;
  float* sgd_v;
  float sgd_lr, sgd_mom;
  __nv_bfloat16* sgd_shadow;
  int sgd_ld_shadow, sgd_shadow_rows;
  int tma_store;  // epilogue writes C through the tmC tensor map
  int a_alt;      // step programs: odd steps read A through the alternate tensor map
};

// Epilogue of the fused attention preprocessing ("Full-Depth MLP Megakernel +
// Fused Attention Preprocessing", "What Worked" and "What Didn't Work": QK
// RMSNorm, partial RoPE and the q gain after the QKV projection, fused in raw
// CUDA).  The accumulator row of a token holds its heads of 64 columns:
// query heads [0, n_q), key heads [n_q, n_qk), then value heads.
struct AttnEpi {
  const float* rstd;    // [M] input RMSNorm scale of each token
  const float* q_gain;  // [n_q]
  int n_q, n_qk;
  int seq_len;          // the position of token m is m % seq_len
  float eps;            // of the QK norm
  float theta;          // RoPE base
};

// sin and cos of a RoPE angle a = pos * f, through the hardware sine and
// cosine approximations directly.  Their reduction of the argument (a scaled
// by 1 / (2 pi) in fp32) loses about |a| 2^-24 rad, some 1e-4 rad for the
// angles below 1,024 rad of sequences of 1,024 positions: the same order as
// the fp32 rounding of the product pos * f itself, and far below the bf16
// rounding of the rotated outputs.
__device__ __forceinline__ void rope_sincos(float a, float& sn, float& cs) {
  __sincosf(a, &sn, &cs);
}

// The RoPE rotation of one token: sin and cos of pos * f_i for the R/2 pairs,
// f_i = theta^(-2i/R) (the same for every token: computed once per CTA into
// shared memory), the same for every query and key head of the token.  For R
// up to 32 they are computed once per tile and kept in registers for the
// warp's heads; for R = 64 (32 pairs) each head computes them again (keeping
// 64 more registers live would spill).
template <int R>
struct RopeAngles {
  static constexpr bool kept = R <= 32;
  float sn[kept ? R / 2 : 1], cs[kept ? R / 2 : 1];
  float pos;
  const float* freq;  // shared memory, R/2 values
};

__device__ __forceinline__ float rope_freq(int i, int R, float log2_theta) {
  return exp2f(-(float)(2 * i) / (float)R * log2_theta);
}

template <int R>
__device__ __forceinline__ void rope_angles(float pos, const float* freq, RopeAngles<R>& ra) {
  ra.pos = pos;
  ra.freq = freq;
  if constexpr (RopeAngles<R>::kept) {
#pragma unroll
    for (int i = 0; i < R / 2; ++i) rope_sincos(pos * freq[i], ra.sn[i], ra.cs[i]);
  }
}

// One head of one token, 64 accumulator values (va: columns 0-31, vb: 32-63)
// before the token's RMSNorm factor rs: rotates the pairs (i, i + R/2) for
// i < R/2 by the token's angles (rotate-half RoPE on the first R dims) in
// place and returns the one factor that finishes the head, rs / RMS(rs v) *
// gain (RoPE is a rotation, so scaling before or after it is the same).  The
// sum of squares runs in four interleaved partial sums, added pairwise.  R is
// a compile-time constant so the partner of every element is a fixed register.
template <int R>
__device__ __forceinline__ float attn_head(float (&va)[32], float (&vb)[32], float rs, float gain,
                                           const RopeAngles<R>& ra, float eps) {
  static_assert(R % 2 == 0 && R <= 64, "rope dims");
  float ss4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 32; ++j) ss4[j & 3] = fmaf(va[j], va[j], ss4[j & 3]);
#pragma unroll
  for (int j = 0; j < 32; ++j) ss4[j & 3] = fmaf(vb[j], vb[j], ss4[j & 3]);
  const float ss = (ss4[0] + ss4[1]) + (ss4[2] + ss4[3]);
  const float inv = 1.0f / sqrtf(rs * rs * ss * (1.0f / 64.0f) + eps);
#pragma unroll
  for (int i = 0; i < R / 2; ++i) {
    constexpr int H = R / 2;
    float& x1 = i < 32 ? va[i] : vb[i - 32];
    float& x2 = i + H < 32 ? va[i + H] : vb[i + H - 32];
    float sn, cs;
    if constexpr (RopeAngles<R>::kept) {
      sn = ra.sn[i];
      cs = ra.cs[i];
    } else {
      rope_sincos(ra.pos * ra.freq[i], sn, cs);
    }
    const float a = x1, b = x2;
    x1 = a * cs - b * sn;
    x2 = b * cs + a * sn;
  }
  return rs * inv * gain;
}

template <int BN, int STAGES>
struct Layout {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // barriers (256 B, padded to keep what follows 1024-aligned), then the
  // optional epilogue staging for TMA stores: per epilogue warp two 32 x 32
  // buffers of up to 4 KiB (fp32); launches without TMA stores do not
  // allocate it, which leaves more of the SM's memory to L1.
  static constexpr int BAR_BYTES = 1024;
  static constexpr int STG_BYTES = 4 * 2 * 4096;
  static constexpr int SMEM_BASE = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
  static constexpr int SMEM = SMEM_BASE + STG_BYTES;
  static constexpr uint32_t TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
};

// Grouped raster: 8 tile-rows at a time sweep all tile-columns, so CTAs that
// run together share A row-blocks and B column-blocks in L2.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int& tm, int& tn) {
  constexpr int G = 8;
  const int group = t / (G * tiles_n);
  const int first = group * G;
  const int gm = min(tiles_m - first, G);
  const int r = t - group * G * tiles_n;
  tm = first + r % gm;
  tn = r / gm;
}

// Bias of columns [n0, n0 + 32) staged in a warp's 32-float shared-memory
// slot (0 past N): one coalesced load per piece instead of 32 broadcast
// loads per thread.  Called by the whole warp at a warp-uniform point.
__device__ __forceinline__ const float* stage_bias(const TcParams& p, int n0, float* slot,
                                                   int lane) {
  if (!p.bias) return nullptr;
  __syncwarp();  // the previous piece's readers are done with the slot
  slot[lane] = n0 + lane < p.N ? __ldg(p.bias + n0 + lane) : 0.f;
  __syncwarp();
  return slot;
}

// The ReLU-mask piece of row m, columns [n0, n0 + 32), loaded ahead of the
// accumulator read so that its latency overlaps the tensor-memory load
// (vector form only for whole, 16-byte aligned pieces).
struct MaskPiece {
  uint4 q[4];
  int vec;
};

__device__ __forceinline__ void load_mask(const TcParams& p, int m, int n0, MaskPiece& mp) {
  mp.vec = 0;
  if (!p.mask || m >= p.M) return;
  const __nv_bfloat16* mrow = p.mask + (size_t)m * p.ldm + n0;
  if (n0 + 32 <= p.N && ((reinterpret_cast<uintptr_t>(mrow) & 15) == 0)) {
#pragma unroll
    for (int q = 0; q < 4; ++q) mp.q[q] = __ldg(reinterpret_cast<const uint4*>(mrow) + q);
    mp.vec = 1;
  }
}

// Bias value for lane `lane` of the 32-column piece at n0, loaded before the
// accumulator is ready; stage_bias_reg publishes it in the warp's slot.
__device__ __forceinline__ float load_bias_lane(const TcParams& p, int n0, int lane) {
  return (p.bias && n0 + lane < p.N) ? __ldg(p.bias + n0 + lane) : 0.f;
}
__device__ __forceinline__ const float* stage_bias_reg(const TcParams& p, float b, float* slot,
                                                       int lane) {
  if (!p.bias) return nullptr;
  __syncwarp();
  slot[lane] = b;
  __syncwarp();
  return slot;
}

// Epilogue arithmetic of one 32-column piece of row m in fp32: + bias (from
// the staged slot, if any), ReLU, ReLU mask (keep where the stored
// activation is > 0).
__device__ __forceinline__ void epilogue_values(const TcParams& p, int m, int n0,
                                                const uint32_t (&r)[32], const float* sb,
                                                const MaskPiece& mp, float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
  if (sb) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 b4 = reinterpret_cast<const float4*>(sb)[q];
      v[4 * q] += b4.x;
      v[4 * q + 1] += b4.y;
      v[4 * q + 2] += b4.z;
      v[4 * q + 3] += b4.w;
    }
  }
  if (p.act == MLP_ACT_RELU) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = fmaxf(v[j], 0.f);
  }
  if (p.mask && m < p.M) {
    const __nv_bfloat16* mrow = p.mask + (size_t)m * p.ldm + n0;
    if (mp.vec) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __nv_bfloat16* mb = reinterpret_cast<const __nv_bfloat16*>(&mp.q[q]);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[q * 8 + e] = bf16_to_f32(mb[e]) > 0.f ? v[q * 8 + e] : 0.f;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n0 + j < p.N) v[j] = bf16_to_f32(mrow[j]) > 0.f ? v[j] : 0.f;
    }
  }
}

// Register store of one piece (outputs whose rows are not 16-byte aligned).
template <int H16>
__device__ __forceinline__ void epilogue_store_regs(const TcParams& p, int m, int n0,
                                                    const float (&v)[32]) {
  const bool full = (n0 + 32 <= p.N);
  if (p.c_bf16) {
    __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(p.C) + (size_t)m * p.ldc + n0;
    if (full && ((reinterpret_cast<uintptr_t>(crow) & 15) == 0)) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 o;
        o.x = pack16x2<H16>(v[q * 8 + 0], v[q * 8 + 1]);
        o.y = pack16x2<H16>(v[q * 8 + 2], v[q * 8 + 3]);
        o.z = pack16x2<H16>(v[q * 8 + 4], v[q * 8 + 5]);
        o.w = pack16x2<H16>(v[q * 8 + 6], v[q * 8 + 7]);
        reinterpret_cast<uint4*>(crow)[q] = o;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n0 + j < p.N) {
          if constexpr (H16) reinterpret_cast<uint16_t*>(crow)[j] = f32_to_16<1>(v[j]);
          else crow[j] = f32_to_bf16(v[j]);
        }
    }
  } else {
    float* crow = static_cast<float*>(p.C) + (size_t)m * p.ldc + n0;
    if (full && ((reinterpret_cast<uintptr_t>(crow) & 15) == 0)) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        reinterpret_cast<float4*>(crow)[q] =
            make_float4(v[q * 4 + 0], v[q * 4 + 1], v[q * 4 + 2], v[q * 4 + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n0 + j < p.N) crow[j] = v[j];
    }
  }
}

// Row `lane` of a warp's 32 x 32 staging box, in the swizzled layout the
// output tensor map uses: 16-byte chunk q of a row is stored at chunk
// q ^ (lane & 7) for fp32 (128-byte rows, 128-byte swizzle) and at
// q ^ ((lane >> 1) & 3) for bf16 (64-byte rows, 64-byte swizzle).
template <int H16>
__device__ __forceinline__ void epilogue_stage_row(uint8_t* box, int c_bf16, int lane,
                                                   const float (&v)[32]) {
  if (c_bf16) {
    uint8_t* row = box + lane * 64;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 o;
      o.x = pack16x2<H16>(v[q * 8 + 0], v[q * 8 + 1]);
      o.y = pack16x2<H16>(v[q * 8 + 2], v[q * 8 + 3]);
      o.z = pack16x2<H16>(v[q * 8 + 4], v[q * 8 + 5]);
      o.w = pack16x2<H16>(v[q * 8 + 6], v[q * 8 + 7]);
      *reinterpret_cast<uint4*>(row + ((q ^ ((lane >> 1) & 3)) << 4)) = o;
    }
  } else {
    uint8_t* row = box + lane * 128;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      *reinterpret_cast<float4*>(row + ((q ^ (lane & 7)) << 4)) =
          make_float4(v[q * 4 + 0], v[q * 4 + 1], v[q * 4 + 2], v[q * 4 + 3]);
  }
}

// Momentum SGD ("Capstone 5: train a network with your CUDA kernels", "Read
// the worked reference": v <- m v - lr g, w <- w + v, also storing g and
// bf16(w)) on the 32 x 32 piece rows [row0, row0 + 32), columns
// [n0, n0 + 32) of a warp.  The fp32
// gradient piece goes through the warp's shared-memory slot (32 x 33 floats,
// conflict-free both ways) so that g, w, v and the bf16 shadow are read and
// written one row at a time across the lanes: 128-byte accesses instead of
// 32 rows touched by every instruction.  Called by the whole warp.
template <int H16>
__device__ __forceinline__ void sgd_epilogue_staged(const TcParams& p, int row0, int n0,
                                                    const uint32_t (&r)[32], float* slot,
                                                    int lane) {
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 32; ++j) slot[lane * 33 + j] = __uint_as_float(r[j]);
  __syncwarp();
  const int n = n0 + lane;
  const bool col_ok = n < p.N;
  // half a piece at a time: its 32 loads in flight at once, then the updates
#pragma unroll
  for (int h = 0; h < 32; h += 16) {
    float wv[16], vv[16];
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
      const int m = row0 + h + rr;
      const size_t off = (size_t)m * p.ldc + n;
      const bool ok = col_ok && m < p.M;
      wv[rr] = ok ? p.sgd_w[off] : 0.f;
      vv[rr] = ok ? p.sgd_v[off] : 0.f;
    }
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
      const int m = row0 + h + rr;
      if (col_ok && m < p.M) {
        const float g = slot[(h + rr) * 33 + lane];
        const size_t off = (size_t)m * p.ldc + n;
        const float nv = p.sgd_mom * vv[rr] - p.sgd_lr * g;
        const float nw = wv[rr] + nv;
        static_cast<float*>(p.C)[off] = g;
        p.sgd_v[off] = nv;
        p.sgd_w[off] = nw;
        if (p.sgd_shadow && m < p.sgd_shadow_rows) {
          if constexpr (H16)
            reinterpret_cast<uint16_t*>(p.sgd_shadow)[(size_t)m * p.sgd_ld_shadow + n] =
                f32_to_16<1>(nw);
          else p.sgd_shadow[(size_t)m * p.sgd_ld_shadow + n] = f32_to_bf16(nw);
        }
      }
    }
  }
}

// The SGD state (w, v) of a warp's 32 rows x 64 columns of a tile, copied
// into shared memory ([32][64] floats each) with cp.async while the tile's
// MMAs run; 16-byte copies where a row segment is whole and aligned, else
// per element (zero-filled outside the matrix).  Completed by cp.async.wait_all.
__device__ __forceinline__ void sgd_state_prefetch(const TcParams& p, int row0, int n_base,
                                                   float* w_s, float* v_s, int lane) {
  const int m = row0 + lane;
  const bool vec = (p.ldc & 3) == 0 && (reinterpret_cast<uintptr_t>(p.sgd_w) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(p.sgd_v) & 15) == 0;
  float* wr = w_s + lane * 64;
  float* vr = v_s + lane * 64;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int n = n_base + 4 * q;
    if (n >= p.N || m >= p.M) break;  // rows past M and columns past N are never read
    const size_t off = (size_t)m * p.ldc + n;
    if (vec && m < p.M && n + 3 < p.N) {
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ptx::smem_u32(wr + 4 * q)),
                   "l"(p.sgd_w + off)
                   : "memory");
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ptx::smem_u32(vr + 4 * q)),
                   "l"(p.sgd_v + off)
                   : "memory");
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool ok = m < p.M && n + e < p.N;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                         ptx::smem_u32(wr + 4 * q + e)),
                     "l"(ok ? p.sgd_w + off + e : p.sgd_w), "r"(ok ? 4 : 0)
                     : "memory");
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                         ptx::smem_u32(vr + 4 * q + e)),
                     "l"(ok ? p.sgd_v + off + e : p.sgd_v), "r"(ok ? 4 : 0)
                     : "memory");
      }
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Momentum SGD as in sgd_epilogue_staged, with w and v of the piece taken
// from the shared-memory copy (columns c0 .. c0 + 31 of the warp's rows).
template <int H16>
__device__ __forceinline__ void sgd_epilogue_smem(const TcParams& p, int row0, int n0, int c0,
                                                  const uint32_t (&r)[32], float* slot,
                                                  const float* w_s, const float* v_s, int lane) {
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 32; ++j) slot[lane * 33 + j] = __uint_as_float(r[j]);
  __syncwarp();
  const int n = n0 + lane;
  const bool col_ok = n < p.N;
  // eight rows at a time: all shared-memory reads of the batch before any of
  // its global stores (the compiler cannot move a load past a store through
  // a pointer it cannot tell apart), so the row chains overlap
#pragma unroll 1
  for (int r0 = 0; r0 < 32; r0 += 8) {
    float g[8], nv[8], nw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = r0 + i;
      g[i] = slot[rr * 33 + lane];
      nv[i] = v_s[rr * 64 + c0 + lane];
      nw[i] = w_s[rr * 64 + c0 + lane];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      nv[i] = p.sgd_mom * nv[i] - p.sgd_lr * g[i];
      nw[i] = nw[i] + nv[i];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int m = row0 + r0 + i;
      if (col_ok && m < p.M) {
        const size_t off = (size_t)m * p.ldc + n;
        static_cast<float*>(p.C)[off] = g[i];
        p.sgd_v[off] = nv[i];
        p.sgd_w[off] = nw[i];
        if (p.sgd_shadow && m < p.sgd_shadow_rows) {
          if constexpr (H16)
            reinterpret_cast<uint16_t*>(p.sgd_shadow)[(size_t)m * p.sgd_ld_shadow + n] =
                f32_to_16<1>(nw[i]);
          else p.sgd_shadow[(size_t)m * p.sgd_ld_shadow + n] = f32_to_bf16(nw[i]);
        }
      }
    }
  }
}

// Softmax cross entropy of one row of at most 32 logits held by one thread
// (the row routine of xent_row.cuh, shared with the one-row-per-thread loss
// kernel).  Writes the fp32 logits (if C is set), 16-bit dZ = (softmax -
// onehot) / norm padded with zeros to xent_ldd, and the argmax (lowest index
// among ties); returns the row loss.
template <int NC, int H16>
__device__ __forceinline__ float xent_epilogue_row_nc(const TcParams& p, int m,
                                                      const uint32_t (&r)[32], const int* labels,
                                                      int* argmax) {
  const int y = __ldg(labels + m);
  float z[NC];
#pragma unroll
  for (int j = 0; j < NC; ++j)
    z[j] = j < p.N ? __uint_as_float(r[j]) + (p.bias ? __ldg(p.bias + j) : 0.f) : 0.f;
  if (p.C) {
    float* lrow = static_cast<float*>(p.C) + (size_t)m * p.ldc;
    if ((reinterpret_cast<uintptr_t>(lrow) & 7) == 0) {
#pragma unroll
      for (int j = 0; j < NC; j += 2) {
        if (j + 1 < p.N) *reinterpret_cast<float2*>(lrow + j) = make_float2(z[j], z[j + 1]);
        else if (j < p.N) lrow[j] = z[j];
      }
    } else {
#pragma unroll
      for (int j = 0; j < NC; ++j)
        if (j < p.N) lrow[j] = z[j];
    }
  }
  float d[NC];
  int am;
  const float loss = xent_row_small<NC>(z, p.N, y, 1.0f / (float)p.xent_norm, d, am);
  __nv_bfloat16* drow = p.xent_dlog + (size_t)m * p.xent_ldd;
  if ((p.xent_ldd & 7) == 0 && (reinterpret_cast<uintptr_t>(drow) & 15) == 0) {
    // rows of a multiple of 8 bf16: 16-byte stores
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (8 * q < p.xent_ldd) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 8 * q + e < NC ? d[(8 * q + e) % NC] : 0.f;
        reinterpret_cast<uint4*>(drow)[q] =
            make_uint4(pack16x2<H16>(v[0], v[1]), pack16x2<H16>(v[2], v[3]),
                       pack16x2<H16>(v[4], v[5]), pack16x2<H16>(v[6], v[7]));
      }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < p.xent_ldd) {
        if constexpr (H16)
          reinterpret_cast<uint16_t*>(drow)[j] = f32_to_16<1>(j < NC ? d[j % NC] : 0.f);
        else drow[j] = f32_to_bf16(j < NC ? d[j % NC] : 0.f);
      }
  }
  if (argmax) argmax[m] = am;
  return loss;
}

template <int H16>
__device__ __forceinline__ float xent_epilogue_row(const TcParams& p, int m,
                                                   const uint32_t (&r)[32], const int* labels,
                                                   int* argmax) {
  return p.N <= 16 ? xent_epilogue_row_nc<16, H16>(p, m, r, labels, argmax)
                   : xent_epilogue_row_nc<32, H16>(p, m, r, labels, argmax);
}

// L1 prefetch of what the epilogue of row m, columns [n0, n0 + bn) will
// read (bias, labels, ReLU mask, the SGD state), issued while the MMAs of
// the tile still run so the epilogue does not wait on L2 or HBM latency.
__device__ __forceinline__ void epilogue_prefetch(const TcParams& p, int m, int n0, int bn,
                                                  int lane, const int* labels) {
  if (p.bias && lane == 0)
    for (int c = 0; c < bn && n0 + c < p.N; c += 32) ptx::prefetch_l1(p.bias + n0 + c);
  if (m >= p.M) return;
  if (labels) ptx::prefetch_l1(labels + m);
  if (p.mask)
    for (int c = 0; c < bn && n0 + c < p.N; c += 64)
      ptx::prefetch_l1(static_cast<const __nv_bfloat16*>(p.mask) + (size_t)m * p.ldm + n0 + c);
  if (p.sgd_w)
    for (int c = 0; c < bn && n0 + c < p.N; c += 32) {
      ptx::prefetch_l1(p.sgd_w + (size_t)m * p.ldc + n0 + c);
      ptx::prefetch_l1(p.sgd_v + (size_t)m * p.ldc + n0 + c);
    }
}

template <int BN, int STAGES, int H16>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcParams p) {
  using L = Layout<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ float xent_part[4];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * L::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * L::B_BYTES);
  uint8_t* stg = sB + STAGES * L::B_BYTES + L::BAR_BYTES;  // epilogue staging (1024-aligned)
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint64_t* xent_bar = done + 1;   // the four epilogue warps' loss partials are in xent_part
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xent_bar + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // per epilogue warp 32 staged bias values, in the upper half of the barrier area
  float* sbias = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 512);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 4);
    }
    ptx::mbar_init(done, 1);
    ptx::mbar_init(xent_bar, 4);
    *s_abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tmA);
    ptx::prefetch_tensormap(&tmB);
    if (p.tma_store) ptx::prefetch_tensormap(&tmC);
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, L::TMEM_COLS);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // prologue done: from here on global memory is touched
  pdl_wait();
  pdl_launch_dependents();

  // stage bookkeeping of the producer, used to drain copies in flight after
  // an abort
  int last_parity[STAGES];

  if (warp == 0) {
    if (lane == 0) {
      for (int s = 0; s < STAGES; ++s) last_parity[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      for (int u = blockIdx.x; u < p.num_tiles * p.splits && !*s_abort; u += gridDim.x) {
        int tm, tn;
        tile_coords(u / p.splits, p.tiles_m, p.tiles_n, tm, tn);
        const int kb0 = (u % p.splits) * p.kb_per_split;
        const int kb1 = min(p.k_blocks, kb0 + p.kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1, p.wait_ns, p.err,
                                      DEVERR_TIMEOUT_PRODUCER)) {
            *s_abort = 1;
            break;
          }
          // 64-wide boxes entirely past M (A M-major) or N (B N-major) are
          // not loaded: they only feed accumulator rows / columns that are
          // never stored, and a box of nothing but fill is slow to deliver
          const bool a_hi = !p.a_mn || tm * BM + 64 < p.M;
          uint32_t bytes = L::STAGE_BYTES - (a_hi ? 0u : 8192u);
          if (p.b_mn) {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              if (tn * BN + j * 64 >= p.N) bytes -= 8192u;
          }
          ptx::mbar_arrive_expect_tx(&full[stage], bytes);
          last_parity[stage] = (int)phase;
          const int k0 = kb * BK;
          uint8_t* a_dst = sA + stage * L::A_BYTES;
          uint8_t* b_dst = sB + stage * L::B_BYTES;
          if (!p.a_mn) {
            ptx::tma_load_2d(a_dst, &tmA, &full[stage], k0, tm * BM);
          } else {
            ptx::tma_load_2d(a_dst, &tmA, &full[stage], tm * BM, k0);
            if (a_hi) ptx::tma_load_2d(a_dst + 8192, &tmA, &full[stage], tm * BM + 64, k0);
          }
          if (!p.b_mn) {
            ptx::tma_load_2d(b_dst, &tmB, &full[stage], k0, tn * BN);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              if (tn * BN + j * 64 < p.N)
                ptx::tma_load_2d(b_dst + j * 8192, &tmB, &full[stage], tn * BN + j * 64, k0);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_16_f32<H16>(BM, BN, p.a_mn, p.b_mn);
      const uint32_t a_lbo = p.a_mn ? 8192u : 16u;
      const uint32_t b_lbo = p.b_mn ? 8192u : 16u;
      const uint32_t a_kstep = p.a_mn ? 2048u : 32u;  // bytes per 16-element k step
      const uint32_t b_kstep = p.b_mn ? 2048u : 32u;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int u = blockIdx.x; u < p.num_tiles * p.splits && !*s_abort; u += gridDim.x) {
        if (!ptx::mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, p.wait_ns, p.err, DEVERR_TIMEOUT_MMA)) {
          *s_abort = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        const int kb0 = (u % p.splits) * p.kb_per_split;
        const int kb1 = min(p.k_blocks, kb0 + p.kb_per_split);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait_bounded(&full[stage], phase, p.wait_ns, p.err, DEVERR_TIMEOUT_MMA)) {
            *s_abort = 1;
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_base = ptx::smem_u32(sA + stage * L::A_BYTES);
          const uint32_t b_base = ptx::smem_u32(sB + stage * L::B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = ptx::sw128_desc(a_base + k * a_kstep, a_lbo, 1024);
            const uint64_t bd = ptx::sw128_desc(b_base + k * b_kstep, b_lbo, 1024);
            ptx::mma_bf16(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          }
          ptx::mma_commit(&empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        ptx::mma_commit(&tfull[acc]);
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      // all MMAs issued by this thread have completed once `done` fires
      ptx::mma_commit(done);
      ptx::mbar_wait_bounded(done, 0, p.wait_ns, p.err, DEVERR_TIMEOUT_TEARDOWN);
    }
  } else {
    const int quarter = warp & 3;  // tensor-memory lanes [32*quarter, 32*quarter + 32)
    const int row = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    int stg_count = 0;  // staged boxes issued by this warp
    for (int u = blockIdx.x; u < p.num_tiles * p.splits; u += gridDim.x) {
      if (*s_abort) break;
      int tm, tn;
      tile_coords(u / p.splits, p.tiles_m, p.tiles_n, tm, tn);
      const int m = tm * BM + row;
      epilogue_prefetch(p, m, tn * BN, BN, lane, p.xent_labels);
      if (!ptx::mbar_wait_bounded(&tfull[acc], acc_phase, p.wait_ns, p.err, DEVERR_TIMEOUT_EPILOGUE)) {
        *s_abort = 1;
        break;
      }
      ptx::tc_fence_after();
      float* part = p.splits > 1 ? p.partial + (size_t)(u % p.splits) * p.M * p.ldp : nullptr;
      float row_loss = 0.f;
      for (int c0 = 0; c0 < BN; c0 += 32) {
        const int n0 = tn * BN + c0;
        if (n0 >= p.N) break;  // warp-uniform
        MaskPiece mp;
        load_mask(p, m, n0, mp);
        uint32_t r[32];
        __syncwarp();
        ptx::tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                    (uint32_t)(acc * BN + c0),
                                r);
        ptx::tmem_ld_wait();
        const float* sb = stage_bias(p, n0, sbias + (warp - 2) * 32, lane);
        if (p.sgd_w) {
          sgd_epilogue_staged<H16>(p, tm * BM + quarter * 32, n0, r,
                              reinterpret_cast<float*>(stg + (warp - 2) * 8192), lane);
        } else if (m < p.M) {
          if (part) {
            float* prow = part + (size_t)m * p.ldp + n0;
            if (n0 + 32 <= p.N) {
#pragma unroll
              for (int q = 0; q < 8; ++q)
                reinterpret_cast<float4*>(prow)[q] =
                    make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
            } else {
              // fully unrolled with a predicate: a loop with a data-dependent
              // trip count would index r[] dynamically and put the whole
              // accumulator piece in local memory on every path
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (n0 + j < p.N) prow[j] = __uint_as_float(r[j]);
            }
          } else if (p.xent_labels) {
            row_loss = xent_epilogue_row<H16>(p, m, r, p.xent_labels, p.xent_argmax);
          } else if (!p.tma_store) {
            float v[32];
            epilogue_values(p, m, n0, r, sb, mp, v);
            epilogue_store_regs<H16>(p, m, n0, v);
          }
        }
        if (p.tma_store) {
          // all lanes take part: rows past M are staged too and clipped by TMA
          float v[32];
          epilogue_values(p, m, n0, r, sb, mp, v);
          uint8_t* box = stg + (warp - 2) * 8192 + (stg_count & 1) * 4096;
          if (stg_count >= 2) {
            if (lane == 0) ptx::bulk_wait_group_read<1>();
            __syncwarp();
          }
          epilogue_stage_row<H16>(box, p.c_bf16, lane, v);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(&tmC, box, n0, tm * BM + quarter * 32);
            ptx::bulk_commit_group();
          }
          ++stg_count;
        }
      }
      if (p.xent_labels) {
        // mean loss of the (single) tile: butterfly sum within each warp,
        // then the four warps in lane-quarter order
        float v = m < p.M ? row_loss : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) {
          xent_part[quarter] = v;
          ptx::mbar_arrive(xent_bar);
        }
        if (warp == 2 && lane == 0 &&
            ptx::mbar_wait_bounded(xent_bar, 0, p.wait_ns, p.err, DEVERR_TIMEOUT_EPILOGUE))
          *p.xent_loss = (((xent_part[0] + xent_part[1]) + xent_part[2]) + xent_part[3]) /
                         (float)p.xent_norm;
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    // the bulk stores must finish before the CTA (and its shared memory) ends
    if (lane == 0) ptx::bulk_wait_group<0>();
    __syncwarp();
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (*s_abort && warp == 0 && lane == 0) {
    // wait (bounded) for TMA copies that may still be landing in shared memory
    for (int s = 0; s < STAGES; ++s)
      if (last_parity[s] >= 0)
        ptx::mbar_wait_bounded(&full[s], (uint32_t)last_parity[s], p.wait_ns, p.err,
                               DEVERR_TIMEOUT_TEARDOWN);
  }
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ step programs
//
// A training step of a small MLP is a chain of small GEMMs, each of which is
// latency-bound (microseconds of TMA round trips and epilogue for a few
// MFLOP).  A step program runs the whole chain in ONE cooperative launch:
// the same warp roles as tc_gemm_kernel, a persistent CTA per SM, and the
// GEMMs of each phase spread over the CTAs by tile; a grid-wide barrier
// separates phases (a phase only reads what earlier phases wrote).  Phase 0
// may cast the input batch to bf16.  The tensor memory, the mbarrier rings
// and their phase bits live across phases.

constexpr int kStepMaxPhases = kStepMaxGemms + 1;
constexpr int STEP_BN = 64;
constexpr int STEP_STAGES = 5;
// per epilogue warp: the SGD state copy, w and v of 32 rows x 64 columns
constexpr int STEP_SGD_BYTES = 4 * 2 * 32 * 64 * 4;

struct StepPhaseDev {
  int kind;  // 0: GEMM tiles, 1: input cast
  int g0, n_gemm, tiles;
};

struct StepProgram {
  CUtensorMap ta[kStepMaxGemms];
  CUtensorMap tb[kStepMaxGemms];
  CUtensorMap ta_alt[kStepMaxGemms];  // A over the second input buffer (GEMMs with a_alt)
  TcParams gp[kStepMaxGemms];
  int tile_base[kStepMaxGemms];  // first tile of GEMM g within its phase
  StepPhaseDev ph[kStepMaxPhases];
  int n_phases;
  const void* cast_src;
  int cast_dtype;
  __nv_bfloat16* cast_dst;
  __nv_bfloat16* cast_dst_alt;
  int cast_ahead_phase;  // phase whose idle CTAs cast the next step's input (-1: none)
  int cast_rows, cast_cols, cast_ld;
  unsigned* bar;  // arrival count of the grid barriers (zeroed before each launch)
  unsigned long long wait_ns;
  int* err;
  int n_steps;
  long long cast_stride, label_stride, loss_stride, argmax_stride;
  int xent_g;  // the GEMM with the fused loss (-1: none)
  int n_gemm;
};

// passed by value as the kernel's parameter block (limit 32,764 bytes)
static_assert(sizeof(TcParams) % 4 == 0, "copied as words");
static_assert(sizeof(StepProgram) <= 32000, "step program exceeds the kernel parameter limit");

// Element i of a step's input rows as a float (image bytes scaled to [0, 1]).
__device__ __forceinline__ float step_load_in(const void* src, int dtype, size_t i) {
  if (dtype == MLP_DTYPE_U8) return (float)static_cast<const uint8_t*>(src)[i] / 255.0f;
  if (dtype == MLP_DTYPE_BF16) return bf16_to_f32(static_cast<const __nv_bfloat16*>(src)[i]);
  if (dtype == MLP_DTYPE_F16) return __half2float(static_cast<const __half*>(src)[i]);
  return static_cast<const float*>(src)[i];
}

// Input rows of step `step` -> 16-bit rows of pitch cast_ld at dst (image
// bytes become byte / 255), spread over CTAs [0, n_cta) of those calling it
// (cta = this CTA's index among them); all threads of the CTA take part.
template <int H16>
__device__ __forceinline__ void step_cast(const StepProgram& prog, int step, __nv_bfloat16* dst,
                                          int cta, int n_cta) {
  const long long stride = (long long)n_cta * blockDim.x;
  const long long first = (long long)cta * blockDim.x + threadIdx.x;
  const void* src = static_cast<const uint8_t*>(prog.cast_src) + step * prog.cast_stride;
  if (prog.cast_dtype == MLP_DTYPE_U8 && (prog.cast_cols & 7) == 0 && (prog.cast_ld & 7) == 0 &&
      (reinterpret_cast<uintptr_t>(src) & 7) == 0) {
    // 8 bytes in, 8 bf16 (16 bytes) out per thread and step
    const int vpr = prog.cast_cols / 8;
    const long long n = (long long)prog.cast_rows * vpr;
    for (long long i = first; i < n; i += stride) {
      const int r = (int)(i / vpr), q = (int)(i % vpr);
      const uint2 b = reinterpret_cast<const uint2*>(src)[i];
      const uint8_t* u8 = reinterpret_cast<const uint8_t*>(&b);
      uint4 o;
      o.x = pack16x2<H16>((float)u8[0] / 255.0f, (float)u8[1] / 255.0f);
      o.y = pack16x2<H16>((float)u8[2] / 255.0f, (float)u8[3] / 255.0f);
      o.z = pack16x2<H16>((float)u8[4] / 255.0f, (float)u8[5] / 255.0f);
      o.w = pack16x2<H16>((float)u8[6] / 255.0f, (float)u8[7] / 255.0f);
      reinterpret_cast<uint4*>(dst + (size_t)r * prog.cast_ld)[q] = o;
    }
  } else {
    const long long n = (long long)prog.cast_rows * prog.cast_cols;
    for (long long i = first; i < n; i += stride) {
      const int r = (int)(i / prog.cast_cols), c = (int)(i % prog.cast_cols);
      if constexpr (H16)
        reinterpret_cast<uint16_t*>(dst)[(size_t)r * prog.cast_ld + c] =
            f32_to_16<1>(step_load_in(src, prog.cast_dtype, (size_t)i));
      else
        dst[(size_t)r * prog.cast_ld + c] = f32_to_bf16(step_load_in(src, prog.cast_dtype, (size_t)i));
    }
  }
}

// Grid-wide barrier of the step program (all threads of every CTA call it):
// one device-scope atomic arrival per CTA and polling of the same counter.
// The proxy fences let the next phase's TMA loads (async proxy) see data
// written with ordinary stores; phases hand data over in global memory only,
// so the fences cover that state space alone (a fence over every state space
// cost 5 % of an epoch).  Bounded: on a timeout the error word is set and the
// CTA's abort flag raised.
__device__ __forceinline__ void step_grid_sync(const StepProgram& prog, volatile int* s_abort,
                                               unsigned& passed) {
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncthreads();
  ++passed;  // barriers of this launch so far, the same count in every CTA
  if (threadIdx.x == 0 && !*s_abort) {
    // the arrival count only grows during a launch (zeroed before it): this
    // barrier is complete once it reaches passed * gridDim.x.  The arrival
    // releases this CTA's writes (ordered before it by the CTA barrier
    // above) at device scope; the polls acquire the other CTAs' writes.
    unsigned* count = prog.bar;
    const unsigned target = passed * gridDim.x;
    unsigned seen;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(seen) : "l"(count) : "memory");
    ++seen;
    if (seen < target) {
      const uint64_t t0 = ptx::globaltimer_ns();
      for (int polls = 1;; ++polls) {
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(seen) : "l"(count) : "memory");
        if (seen >= target) break;
        // the timer is read now and then, not on every poll
        if ((polls & 15) == 0 && ptx::globaltimer_ns() - t0 > prog.wait_ns) {
          record_device_error(prog.err, DEVERR_TIMEOUT_GRID);
          *s_abort = 1;
          break;
        }
      }
    }
  }
  __syncthreads();
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// GEMM g of phase ph that owns the phase's tile u, and u's index within it.
__device__ __forceinline__ int step_gemm_of(const int* tile_base, const StepPhaseDev& ph, int u,
                                            int& local) {
  int g = ph.g0;
  for (int k = 1; k < ph.n_gemm; ++k)
    if (u >= tile_base[ph.g0 + k]) g = ph.g0 + k;
  local = u - tile_base[g];
  return g;
}

template <int BN, int STAGES, int H16>
__global__ void __launch_bounds__(kThreads, 1)
    tc_step_kernel(const __grid_constant__ StepProgram prog) {
  using L = Layout<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ float xent_part[4];
  // the program's per-GEMM parameters, tile bases and phases, copied once:
  // reading them from the parameter block through a computed index is a
  // slow load on every use
  __shared__ TcParams s_gp[kStepMaxGemms];
  __shared__ int s_tile_base[kStepMaxGemms];
  __shared__ StepPhaseDev s_ph[kStepMaxPhases];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * L::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * L::B_BYTES);
  uint8_t* stg = sB + STAGES * L::B_BYTES + L::BAR_BYTES;  // per epilogue warp 8 KiB
  float* sgd_state = reinterpret_cast<float*>(stg + L::STG_BYTES);  // per warp w, v [32][64]
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint64_t* xent_bar = done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xent_bar + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* sbias = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 512);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 4);
    }
    ptx::mbar_init(done, 1);
    ptx::mbar_init(xent_bar, 4);
    *s_abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    // the operand descriptors of every GEMM this CTA will load, ahead of use
    for (int phi = 0; phi < prog.n_phases; ++phi) {
      const StepPhaseDev ph = prog.ph[phi];
      if (ph.kind != 0 || (int)blockIdx.x >= ph.tiles) continue;
      for (int g = ph.g0 + lane; g < ph.g0 + ph.n_gemm; g += 32) {
        ptx::prefetch_tensormap(&prog.ta[g]);
        ptx::prefetch_tensormap(&prog.tb[g]);
        if (prog.gp[g].a_alt) ptx::prefetch_tensormap(&prog.ta_alt[g]);
      }
    }
  }
  {
    const int words = prog.n_gemm * (int)(sizeof(TcParams) / 4);
    const uint32_t* src = reinterpret_cast<const uint32_t*>(prog.gp);
    uint32_t* dst = reinterpret_cast<uint32_t*>(s_gp);
    for (int i = threadIdx.x; i < words; i += blockDim.x) dst[i] = src[i];
    for (int i = threadIdx.x; i < prog.n_gemm; i += blockDim.x) s_tile_base[i] = prog.tile_base[i];
    for (int i = threadIdx.x; i < prog.n_phases; i += blockDim.x) s_ph[i] = prog.ph[i];
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, L::TMEM_COLS);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // pipeline positions of the producer and the MMA issuer, and the
  // accumulator hand-off of the MMA issuer and the epilogue, across phases
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  int last_parity[STAGES];
  for (int s = 0; s < STAGES; ++s) last_parity[s] = -1;
  int xent_uses = 0;
  unsigned barriers_passed = 0;

  const int n_total = prog.n_steps * prog.n_phases;
  const bool dbuf = prog.cast_ahead_phase >= 0;
  for (int it = 0; it < n_total && !*s_abort; ++it) {
    const int step = it / prog.n_phases, phi = it % prog.n_phases;
    const StepPhaseDev ph = s_ph[phi];
    bool sync_after = true;
    if (ph.kind == 1) {
      // with two input buffers only the first step casts in a phase of its
      // own; the later ones were cast during the step before
      if (!dbuf || step == 0) step_cast<H16>(prog, step, prog.cast_dst, blockIdx.x, gridDim.x);
      else sync_after = false;
    } else if (warp == 0) {
      if (lane == 0) {
        // ---------------------------------------------------------- producer
        for (int u = blockIdx.x; u < ph.tiles && !*s_abort; u += gridDim.x) {
          int t;
          const int g = step_gemm_of(s_tile_base, ph, u, t);
          // a private copy: a reference would be re-read after every store
          const TcParams p = s_gp[g];
          int tm, tn;
          tile_coords(t, p.tiles_m, p.tiles_n, tm, tn);
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1, prog.wait_ns, prog.err,
                                        DEVERR_TIMEOUT_PRODUCER)) {
              *s_abort = 1;
              break;
            }
            // boxes entirely past M / N are not loaded (see tc_gemm_kernel)
            const bool a_hi = !p.a_mn || tm * BM + 64 < p.M;
            uint32_t bytes = L::STAGE_BYTES - (a_hi ? 0u : 8192u);
            if (p.b_mn) {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j)
                if (tn * BN + j * 64 >= p.N) bytes -= 8192u;
            }
            ptx::mbar_arrive_expect_tx(&full[stage], bytes);
            last_parity[stage] = (int)phase;
            const int k0 = kb * BK;
            uint8_t* a_dst = sA + stage * L::A_BYTES;
            uint8_t* b_dst = sB + stage * L::B_BYTES;
            const CUtensorMap* tma = (p.a_alt && (step & 1)) ? &prog.ta_alt[g] : &prog.ta[g];
            if (!p.a_mn) {
              ptx::tma_load_2d(a_dst, tma, &full[stage], k0, tm * BM);
            } else {
              ptx::tma_load_2d(a_dst, tma, &full[stage], tm * BM, k0);
              if (a_hi) ptx::tma_load_2d(a_dst + 8192, tma, &full[stage], tm * BM + 64, k0);
            }
            if (!p.b_mn) {
              ptx::tma_load_2d(b_dst, &prog.tb[g], &full[stage], k0, tn * BN);
            } else {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j)
                if (tn * BN + j * 64 < p.N)
                  ptx::tma_load_2d(b_dst + j * 8192, &prog.tb[g], &full[stage], tn * BN + j * 64,
                                   k0);
            }
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
          }
        }
        // the next phase's operand descriptors, so its first loads do not
        // wait for a descriptor fetch
        const StepPhaseDev nx = s_ph[(phi + 1) % prog.n_phases];
        if (nx.kind == 0 && (int)blockIdx.x < nx.tiles)
          for (int g = nx.g0; g < nx.g0 + nx.n_gemm; ++g) {
            ptx::prefetch_tensormap(&prog.ta[g]);
            ptx::prefetch_tensormap(&prog.tb[g]);
            if (s_gp[g].a_alt) ptx::prefetch_tensormap(&prog.ta_alt[g]);
          }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ---------------------------------------------------------- MMA issuer
        for (int u = blockIdx.x; u < ph.tiles && !*s_abort; u += gridDim.x) {
          int t;
          const int g = step_gemm_of(s_tile_base, ph, u, t);
          // a private copy: a reference would be re-read after every store
          const TcParams p = s_gp[g];
          const uint32_t idesc = ptx::idesc_16_f32<H16>(BM, BN, p.a_mn, p.b_mn);
          const uint32_t a_lbo = p.a_mn ? 8192u : 16u;
          const uint32_t b_lbo = p.b_mn ? 8192u : 16u;
          const uint32_t a_kstep = p.a_mn ? 2048u : 32u;
          const uint32_t b_kstep = p.b_mn ? 2048u : 32u;
          if (!ptx::mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, prog.wait_ns, prog.err,
                                      DEVERR_TIMEOUT_MMA)) {
            *s_abort = 1;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
          bool ok = true;
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!ptx::mbar_wait_bounded(&full[stage], phase, prog.wait_ns, prog.err,
                                        DEVERR_TIMEOUT_MMA)) {
              *s_abort = 1;
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t a_base = ptx::smem_u32(sA + stage * L::A_BYTES);
            const uint32_t b_base = ptx::smem_u32(sB + stage * L::B_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint64_t ad = ptx::sw128_desc(a_base + k * a_kstep, a_lbo, 1024);
              const uint64_t bd = ptx::sw128_desc(b_base + k * b_kstep, b_lbo, 1024);
              ptx::mma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
            }
            ptx::mma_commit(&empty[stage]);
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          ptx::mma_commit(&tfull[acc]);
          if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
      }
    } else {
      // ------------------------------------------------------------ epilogue
      const int quarter = warp & 3;
      const int row = quarter * 32 + lane;
      for (int u = blockIdx.x; u < ph.tiles; u += gridDim.x) {
        if (*s_abort) break;
        int t;
        const int g = step_gemm_of(s_tile_base, ph, u, t);
        const TcParams p = s_gp[g];  // private copy, as in the other roles
        // the loss GEMM's labels and outputs of this step
        const int* labels = p.xent_labels ? p.xent_labels + step * prog.label_stride : nullptr;
        int* argmax = p.xent_argmax ? p.xent_argmax + step * prog.argmax_stride : nullptr;
        float* loss_out = p.xent_loss ? p.xent_loss + step * prog.loss_stride : nullptr;
        int tm, tn;
        tile_coords(t, p.tiles_m, p.tiles_n, tm, tn);
        const int m = tm * BM + row;
        const int row0 = tm * BM + quarter * 32;
        float* w_s = sgd_state + (warp - 2) * (2 * 32 * 64);
        float* v_s = w_s + 32 * 64;
        // everything the epilogue reads besides the accumulator is requested
        // now, while the tile's MMAs still run
        epilogue_prefetch(p, m, tn * BN, BN, lane, labels);
        if (p.sgd_w) sgd_state_prefetch(p, row0, tn * BN, w_s, v_s, lane);
        float bias_r[BN / 32];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) bias_r[c] = load_bias_lane(p, tn * BN + 32 * c, lane);
        if (!ptx::mbar_wait_bounded(&tfull[acc], acc_phase, prog.wait_ns, prog.err,
                                    DEVERR_TIMEOUT_EPILOGUE)) {
          *s_abort = 1;
          break;
        }
        ptx::tc_fence_after();
        if (p.sgd_w) {
          asm volatile("cp.async.wait_all;" ::: "memory");
          __syncwarp();
        }
        float row_loss = 0.f;
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32) {
          const int n0 = tn * BN + c0;
          if (n0 >= p.N) break;  // warp-uniform
          MaskPiece mp;
          load_mask(p, m, n0, mp);
          uint32_t r[32];
          __syncwarp();
          ptx::tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                      (uint32_t)(acc * BN + c0),
                                  r);
          ptx::tmem_ld_wait();
          if (p.sgd_w) {
            sgd_epilogue_smem<H16>(p, row0, n0, c0, r,
                              reinterpret_cast<float*>(stg + (warp - 2) * 8192), w_s, v_s, lane);
          } else if (p.xent_labels) {
            if (m < p.M) row_loss = xent_epilogue_row<H16>(p, m, r, labels, argmax);
          } else {
            const float* sb = stage_bias_reg(p, bias_r[c0 / 32], sbias + (warp - 2) * 32, lane);
            if (m < p.M) {
              float v[32];
              epilogue_values(p, m, n0, r, sb, mp, v);
              epilogue_store_regs<H16>(p, m, n0, v);
            }
          }
        }
        if (p.xent_labels) {
          float v = m < p.M ? row_loss : 0.f;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) {
            xent_part[quarter] = v;
            ptx::mbar_arrive(xent_bar);
          }
          if (warp == 2 && lane == 0 &&
              ptx::mbar_wait_bounded(xent_bar, (uint32_t)(xent_uses & 1), prog.wait_ns, prog.err,
                                     DEVERR_TIMEOUT_EPILOGUE)) {
            const float loss = (((xent_part[0] + xent_part[1]) + xent_part[2]) + xent_part[3]) /
                               (float)p.xent_norm;
            check_loss_finite(loss, prog.err);
            *loss_out = loss;
          }
          ++xent_uses;
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
    }
    // the next step's input, cast by the CTAs without a tile in this phase
    if (dbuf && phi == prog.cast_ahead_phase && step + 1 < prog.n_steps &&
        (int)blockIdx.x >= ph.tiles)
      step_cast<H16>(prog, step + 1, ((step + 1) & 1) ? prog.cast_dst_alt : prog.cast_dst,
                (int)blockIdx.x - ph.tiles, (int)gridDim.x - ph.tiles);
    if (it + 1 < n_total && sync_after) step_grid_sync(prog, s_abort, barriers_passed);
  }

  // teardown: the MMA issuer's last MMAs are complete before the tensor
  // memory is freed; after an abort, copies still in flight land first
  if (warp == 1 && lane == 0) {
    ptx::mma_commit(done);
    ptx::mbar_wait_bounded(done, 0, prog.wait_ns, prog.err, DEVERR_TIMEOUT_TEARDOWN);
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (*s_abort && warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s)
      if (last_parity[s] >= 0)
        ptx::mbar_wait_bounded(&full[s], (uint32_t)last_parity[s], prog.wait_ns, prog.err,
                               DEVERR_TIMEOUT_TEARDOWN);
  }
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ CTA-pair kernel
//
// A 256 x 256 output tile per CTA pair (cluster of 2) with tcgen05.mma.cta_group::2:
// CTA r of the pair stages rows [128 r, 128 r + 128) of the A tile and columns
// [128 r, 128 r + 128) of the B tile; the even CTA issues the M = 256, N = 256
// MMAs, whose operands come from both CTAs' shared memory and whose
// accumulator rows land in each CTA's own tensor memory (its 128 rows x 256
// columns, two such buffers).  Per SM that is 32 KiB of operands per 64-wide
// k-block for 2 x 128 x 256 x 64 flops, a third less shared-memory traffic
// per flop than a 128 x 256 single-CTA tile, whose operand streams (TMA
// writes plus MMA reads) otherwise bound the tensor pipe.
//
// Barriers: the even CTA's full[s] collects both CTAs' TMA bytes (the odd
// CTA's loads signal it across the pair); the MMA completions of a stage
// arrive on empty[s] in both CTAs; tfull[a] in both CTAs tells the epilogues
// an accumulator is ready; the even CTA's tempty[a] counts the eight
// epilogue warps of the pair that drained it.
constexpr int BN2 = 256;

// 10 warps: TMA producer, MMA issuer, 8 epilogue warps (two per tensor-memory
// lane quadrant, each draining 128 of the 256 accumulator columns)
constexpr int kPairThreads = 320;

// STG_WARP: staging bytes per epilogue warp: 4 KiB (two 32 x 32 bf16 boxes or
// one fp32 box) for the GEMM epilogue, 8 KiB (two 32 x 64 bf16 boxes: a whole
// head per store) for the streamed attention epilogue, 4 KiB (one such box)
// for the attention epilogue with resident weights.  B_RES: k-blocks of B held
// for the whole tile column (0: B streams through the stages with A).
template <int STAGES, int STG_WARP = 4096, int B_RES = 0>
struct Layout2 {
  static constexpr int A_BYTES = 128 * BK * 2;
  static constexpr int B_BYTES = 128 * BK * 2;
  static constexpr int B_BLOCKS = B_RES > 0 ? B_RES : STAGES;
  static constexpr int BAR_BYTES = 2048;        // barriers, then 8 x 32 bias floats at 512
  static constexpr int STG_BYTES = 8 * STG_WARP;
  static constexpr int SMEM_BASE = 1024 + STAGES * A_BYTES + B_BLOCKS * B_BYTES + BAR_BYTES;
  static constexpr int SMEM = SMEM_BASE + STG_BYTES;
};

// Resident-B attention projection: K up to 8 k-blocks (512) of the CTA's 128
// weight columns stay in shared memory while the pair walks down a column of
// tiles, so only the token rows stream (half the operand bytes per tile).
constexpr int kBResBlocks = 8;

template <int STAGES, int EPI, bool BRES>
using PairLayout = Layout2<STAGES, (EPI > 0 && !BRES ? 8192 : 4096), (BRES ? kBResBlocks : 0)>;

// The units (tiles x splits) of one CTA pair: every n_pairs-th unit of the
// grouped raster, or, with resident B, a contiguous run of the column-major
// tile order (a run changes tile column at most a few times, and not at all
// when the pair count is a multiple of the column count).
struct PairUnits {
  int begin, end, stride;
};

__device__ __forceinline__ PairUnits pair_units(int pair, int n_pairs, int units, bool bres) {
  if (!bres) return {pair, units, n_pairs};
  return {(int)((long long)pair * units / n_pairs), (int)((long long)(pair + 1) * units / n_pairs),
          1};
}

__device__ __forceinline__ void pair_tile(const TcParams& p, int u, bool bres, int& tm, int& tn) {
  if (bres) {
    tn = u / p.tiles_m;
    tm = u - tn * p.tiles_m;
  } else {
    tile_coords(u / p.splits, p.tiles_m, p.tiles_n, tm, tn);
  }
}

// EPI = 0: the GEMM epilogue (bias, activation, mask, split-K partials);
// EPI = R > 0: the fused attention preprocessing with R RoPE dims (ae).
template <int STAGES, int H16, int EPI, bool BRES = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const TcParams p,
                        const AttnEpi ae) {
  static_assert(!BRES || EPI > 0, "resident B is the attention projection's");
  using L = PairLayout<STAGES, EPI, BRES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * L::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + L::B_BLOCKS * L::B_BYTES);
  uint8_t* stg = sB + L::B_BLOCKS * L::B_BYTES + L::BAR_BYTES;
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint64_t* bfree = done + 1;  // resident B: the MMAs reading it have completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bfree + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* sbias = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 512);
  float* sfreq = sbias;  // attention: the RoPE frequencies (no bias there)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const int units = p.num_tiles * p.splits;
  const PairUnits ur = pair_units(pair, n_pairs, units, BRES);

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 16);  // the pair's 16 epilogue warps
    }
    ptx::mbar_init(done, 1);
    ptx::mbar_init(bfree, 1);
    *s_abort = 0;
  }
  if constexpr (EPI > 0) {
    if (threadIdx.x < EPI / 2) sfreq[threadIdx.x] = rope_freq(threadIdx.x, EPI, log2f(ae.theta));
  }
  if (warp == 0 && lane == 0) {
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tmA);
    ptx::prefetch_tensormap(&tmB);
    if (p.tma_store) ptx::prefetch_tensormap(&tmC);
  }
  if (warp == 1) ptx::tmem_alloc_pair(tmem_slot, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();

  int last_parity[STAGES];

  if (warp == 0) {
    if (lane == 0) {
      for (int s = 0; s < STAGES; ++s) last_parity[s] = -1;
      const uint32_t full0 = ptx::mapa_shared(ptx::smem_u32(full), 0);  // the even CTA's full[]
      int stage = 0;
      uint32_t phase = 0;
      int b_tn = -1, b_loads = 0;  // resident B: its tile column, and how often it was loaded
      for (int u = ur.begin; u < ur.end && !*s_abort; u += ur.stride) {
        int tm, tn;
        pair_tile(p, u, BRES, tm, tn);
        const int kb0 = (u % p.splits) * p.kb_per_split;
        const int kb1 = min(p.k_blocks, kb0 + p.kb_per_split);
        const int m0 = tm * 256 + (int)rank * 128;
        const int n0 = tn * BN2 + (int)rank * 128;
        // resident B: a new tile column is loaded with this unit's A stages,
        // once the pair's MMAs on the old one have completed
        const bool load_b = !BRES || tn != b_tn;
        if (BRES && load_b) {
          if (b_loads > 0 &&
              !ptx::mbar_wait_cluster_bounded(bfree, (uint32_t)((b_loads - 1) & 1), p.wait_ns,
                                              p.err, DEVERR_TIMEOUT_PRODUCER)) {
            *s_abort = 1;
            break;
          }
          b_tn = tn;
          ++b_loads;
        }
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait_cluster_bounded(&empty[stage], phase ^ 1, p.wait_ns, p.err,
                                              DEVERR_TIMEOUT_PRODUCER)) {
            *s_abort = 1;
            break;
          }
          if (rank == 0) {
            ptx::mbar_arrive_expect_tx(&full[stage],
                                       2 * (L::A_BYTES + (load_b ? L::B_BYTES : 0)));
            last_parity[stage] = (int)phase;
          }
          const uint32_t bar = full0 + (uint32_t)stage * 8u;
          const int k0 = kb * BK;
          uint8_t* a_dst = sA + stage * L::A_BYTES;
          uint8_t* b_dst = sB + (BRES ? kb : stage) * L::B_BYTES;
          if (!p.a_mn) {
            ptx::tma_load_2d_pair(a_dst, &tmA, bar, k0, m0);
          } else {
            ptx::tma_load_2d_pair(a_dst, &tmA, bar, m0, k0);
            ptx::tma_load_2d_pair(a_dst + 8192, &tmA, bar, m0 + 64, k0);
          }
          if (!load_b) {
          } else if (!p.b_mn) {
            ptx::tma_load_2d_pair(b_dst, &tmB, bar, k0, n0);
          } else {
            ptx::tma_load_2d_pair(b_dst, &tmB, bar, n0, k0);
            ptx::tma_load_2d_pair(b_dst + 8192, &tmB, bar, n0 + 64, k0);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      const uint32_t idesc = ptx::idesc_16_f32<H16>(256, BN2, p.a_mn, p.b_mn);
      const uint32_t a_lbo = p.a_mn ? 8192u : 16u;
      const uint32_t b_lbo = p.b_mn ? 8192u : 16u;
      const uint32_t a_kstep = p.a_mn ? 2048u : 32u;
      const uint32_t b_kstep = p.b_mn ? 2048u : 32u;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int u = ur.begin; u < ur.end && !*s_abort; u += ur.stride) {
        if (!ptx::mbar_wait_cluster_bounded(&tempty[acc], acc_phase ^ 1, p.wait_ns, p.err,
                                            DEVERR_TIMEOUT_MMA)) {
          *s_abort = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN2);
        const int kb0 = (u % p.splits) * p.kb_per_split;
        const int kb1 = min(p.k_blocks, kb0 + p.kb_per_split);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait_bounded(&full[stage], phase, p.wait_ns, p.err, DEVERR_TIMEOUT_MMA)) {
            *s_abort = 1;
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_base = ptx::smem_u32(sA + stage * L::A_BYTES);
          const uint32_t b_base = ptx::smem_u32(sB + (BRES ? kb : stage) * L::B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = ptx::sw128_desc(a_base + k * a_kstep, a_lbo, 1024);
            const uint64_t bd = ptx::sw128_desc(b_base + k * b_kstep, b_lbo, 1024);
            ptx::mma_bf16_pair(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          }
          ptx::mma_commit_pair_multicast(&empty[stage], 3);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        ptx::mma_commit_pair_multicast(&tfull[acc], 3);
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        if constexpr (BRES) {
          // the next unit starts a new tile column: both producers may
          // overwrite their B once these MMAs have completed
          if (u + 1 < ur.end && (u + 1) / p.tiles_m != u / p.tiles_m)
            ptx::mma_commit_pair_multicast(bfree, 3);
        }
      }
      ptx::mma_commit_pair_multicast(done, 1);
      ptx::mbar_wait_bounded(done, 0, p.wait_ns, p.err, DEVERR_TIMEOUT_TEARDOWN);
    }
  } else {
    const int quarter = warp & 3;
    const int c_half = ((warp - 2) >> 2) * (BN2 / 2);  // this warp's 128 accumulator columns
    const uint32_t tempty0 = ptx::mapa_shared(ptx::smem_u32(tempty), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    int stg_count = 0;
    for (int u = ur.begin; u < ur.end; u += ur.stride) {
      if (*s_abort) break;
      if (!ptx::mbar_wait_cluster_bounded(&tfull[acc], acc_phase, p.wait_ns, p.err,
                                          DEVERR_TIMEOUT_EPILOGUE)) {
        *s_abort = 1;
        break;
      }
      ptx::tc_fence_after();
      int tm, tn;
      pair_tile(p, u, BRES, tm, tn);
      float* part = p.splits > 1 ? p.partial + (size_t)(u % p.splits) * p.M * p.ldp : nullptr;
      const int row0 = tm * 256 + (int)rank * 128 + quarter * 32;  // this warp's first row
      const int m = row0 + lane;
      if constexpr (EPI == 0) {
        // ReLU-mask pieces are fetched one piece ahead of their use
        MaskPiece mp_next;
        load_mask(p, m, tn * BN2 + c_half, mp_next);
        for (int c0 = c_half; c0 < c_half + BN2 / 2; c0 += 32) {
          const int n0 = tn * BN2 + c0;
          if (n0 >= p.N) break;  // warp-uniform
          const MaskPiece mp = mp_next;
          if (c0 + 32 < c_half + BN2 / 2 && n0 + 32 < p.N) load_mask(p, m, n0 + 32, mp_next);
          uint32_t r[32];
          __syncwarp();
          ptx::tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                      (uint32_t)(acc * BN2 + c0),
                                  r);
          ptx::tmem_ld_wait();
          const float* sb = stage_bias(p, n0, sbias + (warp - 2) * 32, lane);
          if (part) {
            if (m < p.M) {
              float* prow = part + (size_t)m * p.ldp + n0;
              if (n0 + 32 <= p.N) {
  #pragma unroll
                for (int q = 0; q < 8; ++q)
                  reinterpret_cast<float4*>(prow)[q] =
                      make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                  __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
              } else {
                // fully unrolled with a predicate: a loop with a data-dependent
                // trip count would index r[] dynamically and put the whole
                // accumulator piece in local memory on every path
  #pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (n0 + j < p.N) prow[j] = __uint_as_float(r[j]);
              }
            }
          } else if (!p.tma_store) {
            if (m < p.M) {
              float v[32];
              epilogue_values(p, m, n0, r, sb, mp, v);
              epilogue_store_regs<H16>(p, m, n0, v);
            }
          } else if (row0 < p.M) {  // warp-uniform; rows past M are clipped by TMA
            float v[32];
            epilogue_values(p, m, n0, r, sb, mp, v);
            // per warp 4 KiB: two 2 KiB bf16 boxes in turn, or one fp32 box
            uint8_t* box = stg + (warp - 2) * 4096 + (p.c_bf16 ? (stg_count & 1) * 2048 : 0);
            if (p.c_bf16 ? stg_count >= 2 : stg_count >= 1) {
              if (lane == 0) {
                if (p.c_bf16) ptx::bulk_wait_group_read<1>();
                else ptx::bulk_wait_group_read<0>();
              }
              __syncwarp();
            }
            epilogue_stage_row<H16>(box, p.c_bf16, lane, v);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_2d(&tmC, box, n0, row0);
              ptx::bulk_commit_group();
            }
            ++stg_count;
          }
        }
      } else {
        // fused attention preprocessing: one 64-column head per step
        const float rs = m < p.M ? __ldg(ae.rstd + m) : 0.f;
        const float pos = (float)(m < p.M ? m % ae.seq_len : 0);
        // a head's 64 bf16 / fp16 outputs: one 32 x 64 staging box (128-byte
        // rows, 128-byte swizzle) and one TMA store for large outputs, else
        // straight from registers
        auto store_head = [&](float (&va)[32], float (&vb)[32], float sc, int nn) {
          if (!p.tma_store) {
            if (m < p.M) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                va[j] *= sc;
                vb[j] *= sc;
              }
              epilogue_store_regs<H16>(p, m, nn, va);
              epilogue_store_regs<H16>(p, m, nn + 32, vb);
            }
            return;
          }
          if (row0 >= p.M) return;  // warp-uniform; rows past M are clipped by TMA
          // two boxes per warp in turn (streamed weights), or one (resident)
          constexpr int kBoxes = BRES ? 1 : 2;
          uint8_t* box = stg + (warp - 2) * (kBoxes * 4096) + (stg_count % kBoxes) * 4096;
          if (stg_count >= kBoxes) {
            if (lane == 0) ptx::bulk_wait_group_read<kBoxes - 1>();
            __syncwarp();
          }
          uint8_t* row = box + lane * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float* v = q < 4 ? &va[q * 8] : &vb[(q - 4) * 8];
            uint4 o;
            o.x = pack16x2<H16>(v[0] * sc, v[1] * sc);
            o.y = pack16x2<H16>(v[2] * sc, v[3] * sc);
            o.z = pack16x2<H16>(v[4] * sc, v[5] * sc);
            o.w = pack16x2<H16>(v[6] * sc, v[7] * sc);
            *reinterpret_cast<uint4*>(row + ((q ^ (lane & 7)) << 4)) = o;
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(&tmC, box, nn, row0);
            ptx::bulk_commit_group();
          }
          ++stg_count;
        };
        // this token's rotation, computed once for the warp's heads of the tile
        RopeAngles<EPI> angles;
        if (tn * BN2 + c_half < ae.n_qk * 64) rope_angles<EPI>(pos, sfreq, angles);
        // the accumulator goes back to the MMA issuer as soon as this warp's
        // last head of the tile is in registers
        auto release = [&] {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (rank == 0) ptx::mbar_arrive(&tempty[acc]);
            else ptx::mbar_arrive_remote(tempty0 + (uint32_t)acc * 8u);
          }
        };
        bool released = false;
        for (int hc = c_half; hc < c_half + BN2 / 2; hc += 64) {
          const int n0 = tn * BN2 + hc;
          if (n0 >= p.N) break;  // warp-uniform
          uint32_t ra[32], rb[32];
          __syncwarp();
          const uint32_t taddr =
              tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN2 + hc);
          ptx::tmem_ld_32x32b_x32(taddr, ra);
          ptx::tmem_ld_32x32b_x32(taddr + 32, rb);
          ptx::tmem_ld_wait();
          if (hc + 64 >= c_half + BN2 / 2 || n0 + 64 >= p.N) {
            release();
            released = true;
          }
          float va[32], vb[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            va[j] = __uint_as_float(ra[j]);
            vb[j] = __uint_as_float(rb[j]);
          }
          const int head = n0 >> 6;
          float sc = rs;  // value heads: the token's RMSNorm factor only
          if (head < ae.n_qk)  // warp-uniform: query and key heads
            sc = attn_head<EPI>(va, vb, rs, head < ae.n_q ? __ldg(ae.q_gain + head) : 1.0f,
                                angles, ae.eps);
          store_head(va, vb, sc, n0);
        }
        if (!released) release();
      }
      if constexpr (EPI == 0) {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) ptx::mbar_arrive(&tempty[acc]);
          else ptx::mbar_arrive_remote(tempty0 + (uint32_t)acc * 8u);
        }
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    if (lane == 0) ptx::bulk_wait_group<0>();
    __syncwarp();
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (*s_abort && warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s)
      if (last_parity[s] >= 0)
        ptx::mbar_wait_bounded(&full[s], (uint32_t)last_parity[s], p.wait_ns, p.err,
                               DEVERR_TIMEOUT_TEARDOWN);
  }
  __syncwarp();
  __syncthreads();
  // neither CTA frees its tensor memory or leaves while the pair's MMAs or
  // signals may still reach it
  ptx::cluster_sync();
  if (warp == 1) {
    __syncwarp();
    ptx::tmem_dealloc_pair(tmem_base, 512);
  }
}

// Split-K finish: out = epilogue(sum_s partial[s]) in a fixed order, four
// consecutive columns per thread.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const TcParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const long long quads = (long long)p.M * (p.ldp / 4);
  const size_t plane = (size_t)p.M * p.ldp;
  for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < quads;
       q += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(q / (p.ldp / 4));
    const int n0 = (int)(q % (p.ldp / 4)) * 4;
    if (n0 >= p.N) continue;
    float4 acc = __ldcs(reinterpret_cast<const float4*>(p.partial + (size_t)m * p.ldp + n0));
    for (int s = 1; s < p.splits; ++s) {
      const float4 v =
          __ldcs(reinterpret_cast<const float4*>(p.partial + s * plane + (size_t)m * p.ldp + n0));
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    float v[4] = {acc.x, acc.y, acc.z, acc.w};
    for (int j = 0; j < 4 && n0 + j < p.N; ++j) {
      const int n = n0 + j;
      float o = v[j];
      if (p.bias) o += p.bias[n];
      if (p.act == MLP_ACT_RELU) o = fmaxf(o, 0.f);
      if (p.mask) o = bf16_to_f32(p.mask[(size_t)m * p.ldm + n]) > 0.f ? o : 0.f;
      if (p.c_bf16)
        static_cast<uint16_t*>(p.C)[(size_t)m * p.ldc + n] =
            f32_to_16_fmt(o, p.f16 ? MLP_DTYPE_F16 : MLP_DTYPE_BF16);
      else static_cast<float*>(p.C)[(size_t)m * p.ldc + n] = o;
    }
  }
}

template <int BN, int STAGES, int H16>
mlp_status launch_bn(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                     const TcParams& p, cudaStream_t st) {
  using L = Layout<BN, STAGES>;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(tc_gemm_kernel<BN, STAGES, H16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM) != cudaSuccess)
      return MLP_ERR_CUDA;
    configured = true;
  }
  const int units = p.num_tiles * p.splits;
  int grid = units < num_sms() ? units : num_sms();
  {
    static const char* names[3] = {"gemm_tc_bn64", "gemm_tc_bn128", "gemm_tc_bn256"};
    static const char* split_names[3] = {"gemm_tc_splitk_bn64", "gemm_tc_splitk_bn128",
                                         "gemm_tc_splitk_bn256"};
    const int which = BN == 64 ? 0 : (BN == 128 ? 1 : 2);
    LaunchScope ls(p.splits > 1 ? split_names[which] : names[which], st, p.M, p.N, p.K);
    launch_k(tc_gemm_kernel<BN, STAGES, H16>, dim3(grid), dim3(kThreads),
             p.tma_store || p.sgd_w ? L::SMEM : L::SMEM_BASE, st, ta, tb, tc, p);
  }
  MLP_CHECK(launch_status());
  if (p.splits > 1) {
    const long long quads = (long long)p.M * (p.ldp / 4);
    long long blocks = (quads + 255) / 256;
    if (blocks > (long long)num_sms() * 8) blocks = (long long)num_sms() * 8;
    LaunchScope ls("splitk_reduce", st, p.M, p.N, p.splits);
    launch_k(splitk_reduce_kernel, dim3((int)blocks), dim3(256), 0, st, p);
    return launch_status();
  }
  return MLP_OK;
}

template <int STAGES, int H16, int EPI = 0, bool BRES = false>
mlp_status launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                       const TcParams& p, cudaStream_t st, const AttnEpi& ae = AttnEpi{}) {
  using L = PairLayout<STAGES, EPI, BRES>;
  static_assert(L::SMEM <= 232448, "pair kernel shared memory");
  static bool configured = false;
  static int max_pairs = 0;
  if (!configured) {
    if (cudaFuncSetAttribute(tc_gemm_pair_kernel<STAGES, H16, EPI, BRES>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM) != cudaSuccess)
      return MLP_ERR_CUDA;
    // pairs that fit at once (a GPC with an odd number of free SMs leaves one over)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    cfg.blockDim = dim3(kPairThreads);
    cfg.dynamicSmemBytes = L::SMEM;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_pair_kernel<STAGES, H16, EPI, BRES>, &cfg) !=
            cudaSuccess ||
        n < 1) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    max_pairs = n;
    configured = true;
  }
  const int units = p.num_tiles * p.splits;
  const int pairs = units < max_pairs ? units : max_pairs;
  {
    LaunchScope ls(EPI ? "attn_prep_gemm" : (p.splits > 1 ? "gemm_tc_pair_splitk" : "gemm_tc_pair"),
                   st, p.M, p.N, p.K);
    launch_k(tc_gemm_pair_kernel<STAGES, H16, EPI, BRES>, dim3(2 * pairs), dim3(kPairThreads),
             p.tma_store ? L::SMEM : L::SMEM_BASE, st, ta, tb, tc, p, ae);
  }
  MLP_CHECK(launch_status());
  if (p.splits > 1) {
    const long long quads = (long long)p.M * (p.ldp / 4);
    long long blocks = (quads + 255) / 256;
    if (blocks > (long long)num_sms() * 8) blocks = (long long)num_sms() * 8;
    LaunchScope ls("splitk_reduce", st, p.M, p.N, p.splits);
    launch_k(splitk_reduce_kernel, dim3((int)blocks), dim3(256), 0, st, p);
    return launch_status();
  }
  return MLP_OK;
}

// Kernel choice and split-K plan from the shape alone (so workspace sizes do
// not depend on the device).  CTA pairs with 256 x 256 tiles whenever both
// output dimensions exceed 128 and there are enough pair tiles for ~76 pairs
// (unless their last round is so ragged that single-CTA tiles finish first,
// e.g. M = 1025), or K is long enough to split; otherwise single-CTA
// 128 x BN tiles, split only when 128 x 256 tiles leave most of ~144 SMs idle
// and K is long.
struct GemmPlan {
  bool pair;
  int splits, kb_per_split;
};

GemmPlan gemm_plan(int M, int N, int K, bool fused) {
  GemmPlan pl;
  const int kblocks = (K + BK - 1) / BK;
  pl.pair = false;
  int s = 1;
  if (!fused && M > 128 && N > 128) {
    const int pair_tiles = ((M + 255) / 256) * ((N + BN2 - 1) / BN2);
    const int single_tiles = ((M + BM - 1) / BM) * ((N + 255) / 256);
    // rounds of tiles over ~76 pairs vs ~152 single CTAs; a pair round does
    // about 1.25x the work per SM of a single-CTA round in the same time
    const int pair_rounds = (pair_tiles + 75) / 76;
    const int single_rounds = (single_tiles + 151) / 152;
    if (pair_tiles >= 48 && 4 * pair_rounds <= 5 * single_rounds) {
      pl.pair = true;
    } else if (pair_tiles < 48 && kblocks >= 64) {
      s = 76 / pair_tiles;
      if (s > 16) s = 16;
      if (s > kblocks / 16) s = kblocks / 16;
      if (s >= 2) pl.pair = true;
      else s = 1;
    }
  }
  if (!pl.pair && !fused) {
    const int tiles = ((M + BM - 1) / BM) * ((N + 255) / 256);
    if (tiles < 72 && kblocks >= 64) {
      s = 144 / tiles;
      if (s > 16) s = 16;
      if (s > kblocks / 16) s = kblocks / 16;
      if (s < 1) s = 1;
    }
  }
  int per = (kblocks + s - 1) / s;
  s = (kblocks + per - 1) / per;
  pl.splits = s;
  pl.kb_per_split = per;
  return pl;
}

// Kernel parameters and operand tensor maps of one GEMM for a tile grid of
// tiles_m x ceil(N / BN) (K-major B boxes of b_box_rows rows).
mlp_status prepare_tc(const GemmArgs& g, int tiles_m, int BN, int splits, int kb_per_split,
                      int b_box_rows, unsigned long long wait_ns, TcParams* pp, CUtensorMap* ta,
                      CUtensorMap* tb) {
  TcParams& p = *pp;
  p.M = g.M; p.N = g.N; p.K = g.K;
  p.a_alt = 0;
  p.a_mn = g.a_trans ? 1 : 0;       // A stored [K][M]  -> M-major tiles
  p.b_mn = g.b_trans ? 0 : 1;       // B stored [K][N]  -> N-major tiles
  p.tiles_m = tiles_m;
  p.tiles_n = (g.N + BN - 1) / BN;
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.k_blocks = (g.K + BK - 1) / BK;
  p.bias = g.bias;
  p.act = g.act;
  p.mask = static_cast<const __nv_bfloat16*>(g.mask);
  p.ldm = g.ldm;
  p.C = g.C;
  p.ldc = g.ldc;
  p.c_bf16 = g.c_bf16;
  p.f16 = g.f16;
  p.wait_ns = wait_ns;
  p.splits = splits;
  p.kb_per_split = kb_per_split;
  p.ldp = (g.N + 3) / 4 * 4;
  p.partial = splits > 1 ? static_cast<float*>(g.ws) : nullptr;
  p.xent_labels = g.xent_labels;
  p.xent_dlog = static_cast<__nv_bfloat16*>(g.xent_dlog);
  p.xent_ldd = g.xent_ldd;
  p.xent_loss = g.xent_loss;
  p.xent_argmax = g.xent_argmax;
  p.xent_norm = g.xent_norm;
  p.sgd_w = g.sgd_w;
  p.sgd_v = g.sgd_v;
  p.sgd_lr = g.sgd_lr;
  p.sgd_mom = g.sgd_mom;
  p.sgd_shadow = g.sgd_shadow;
  p.sgd_ld_shadow = g.sgd_ld_shadow;
  p.sgd_shadow_rows = g.sgd_shadow_rows;
  p.tma_store = 0;
  if (p.xent_labels && (p.num_tiles != 1 || g.N > 32 || !p.xent_dlog || !p.xent_loss))
    return MLP_ERR_UNSUPPORTED_SHAPE;
  if ((p.xent_labels || p.sgd_w) && splits > 1) return MLP_ERR_UNSUPPORTED_SHAPE;
  p.err = device_error_word();
  if (!p.err) return MLP_ERR_CUDA;

  bool ok;
  if (!p.a_mn)
    ok = encode_tmap_bf16_2d(ta, g.A, g.K, g.M, (unsigned long long)g.lda * 2, 64, BM);
  else
    ok = encode_tmap_bf16_2d(ta, g.A, g.M, g.K, (unsigned long long)g.lda * 2, 64, 64);
  if (!ok) return MLP_ERR_CUDA;
  if (!p.b_mn)
    ok = encode_tmap_bf16_2d(tb, g.B, g.K, g.N, (unsigned long long)g.ldb * 2, 64, b_box_rows);
  else
    ok = encode_tmap_bf16_2d(tb, g.B, g.N, g.K, (unsigned long long)g.ldb * 2, 64, 64);
  if (!ok) return MLP_ERR_CUDA;
  return MLP_OK;
}

}  // namespace

bool step_gemm_supported(const GemmArgs& g) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return false;
  const int tiles = ((g.M + BM - 1) / BM) * ((g.N + STEP_BN - 1) / STEP_BN);
  if (tiles > num_sms()) return false;
  if (g.xent_labels && (g.M > BM || g.N > 32)) return false;
  // one pass over K, accumulator in tensor memory: no split-K
  return true;
}

mlp_status launch_step_program(const StepSpec& s, unsigned* bar_words, unsigned long long wait_ns,
                               cudaStream_t st) {
  using L = Layout<STEP_BN, STEP_STAGES>;
  static bool configured[2] = {false, false};
  const int h16 = s.f16 ? 1 : 0;
  if (!configured[h16]) {
    if (cudaFuncSetAttribute(h16 ? tc_step_kernel<STEP_BN, STEP_STAGES, 1>
                                 : tc_step_kernel<STEP_BN, STEP_STAGES, 0>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::SMEM + STEP_SGD_BYTES) != cudaSuccess)
      return MLP_ERR_CUDA;
    configured[h16] = true;
  }
  if (s.n_gemm < 0 || s.n_gemm > kStepMaxGemms || !bar_words) return MLP_ERR_INVALID_ARG;
  StepProgram prog;  // ~12 KiB of kernel parameters
  memset(&prog, 0, sizeof(prog));
  int np = 0;
  if (s.cast_src && s.cast_rows > 0 && s.cast_cols > 0) {
    prog.ph[np++] = StepPhaseDev{1, 0, 0, 0};
    prog.cast_src = s.cast_src;
    prog.cast_dtype = s.cast_dtype;
    prog.cast_dst = static_cast<__nv_bfloat16*>(s.cast_dst);
    prog.cast_rows = s.cast_rows;
    prog.cast_cols = s.cast_cols;
    prog.cast_ld = s.cast_ld;
  }
  int grid = 1;
  for (int g = 0; g < s.n_gemm; ++g) {
    const GemmArgs& a = s.gemm[g];
    if (!step_gemm_supported(a)) return MLP_ERR_UNSUPPORTED_SHAPE;
    if (g > 0 && s.phase[g] < s.phase[g - 1]) return MLP_ERR_INVALID_ARG;
    MLP_CHECK(prepare_tc(a, (a.M + BM - 1) / BM, STEP_BN, 1, (a.K + BK - 1) / BK, STEP_BN, wait_ns,
                         &prog.gp[g], &prog.ta[g], &prog.tb[g]));
    if (g == 0 || s.phase[g] != s.phase[g - 1]) {
      if (np >= kStepMaxPhases) return MLP_ERR_INVALID_ARG;
      prog.ph[np++] = StepPhaseDev{0, g, 0, 0};
    }
    StepPhaseDev& ph = prog.ph[np - 1];
    prog.tile_base[g] = ph.tiles;
    ph.tiles += prog.gp[g].num_tiles;
    ph.n_gemm += 1;
    if (ph.tiles > grid) grid = ph.tiles;
  }
  if (np == 0) return MLP_OK;
  if (grid > num_sms()) return MLP_ERR_UNSUPPORTED_SHAPE;
  if (s.n_steps < 1) return MLP_ERR_INVALID_ARG;
  // Two input buffers: the next step's input is cast by the CTAs idle in the
  // GEMM phase with the fewest tiles; GEMMs reading the input alternate.
  prog.cast_ahead_phase = -1;
  if (s.cast_dst_alt && s.n_steps > 1 && prog.ph[0].kind == 1) {
    int best = -1;
    for (int i = 1; i < np; ++i)
      if (prog.ph[i].tiles < grid && (best < 0 || prog.ph[i].tiles < prog.ph[best].tiles)) best = i;
    if (best > 0) {
      for (int g = 0; g < s.n_gemm; ++g) {
        if (s.gemm[g].A != s.cast_dst) continue;
        GemmArgs a2 = s.gemm[g];
        a2.A = s.cast_dst_alt;
        TcParams p2;
        CUtensorMap tb2;
        MLP_CHECK(prepare_tc(a2, (a2.M + BM - 1) / BM, STEP_BN, 1, (a2.K + BK - 1) / BK, STEP_BN,
                             wait_ns, &p2, &prog.ta_alt[g], &tb2));
        prog.gp[g].a_alt = 1;
      }
      prog.cast_ahead_phase = best;
      prog.cast_dst_alt = static_cast<__nv_bfloat16*>(s.cast_dst_alt);
    }
  }
  prog.n_phases = np;
  prog.n_steps = s.n_steps;
  prog.cast_stride = s.cast_stride;
  prog.label_stride = s.label_stride;
  prog.loss_stride = s.loss_stride;
  prog.argmax_stride = s.argmax_stride;
  prog.xent_g = -1;
  prog.n_gemm = s.n_gemm;
  for (int g = 0; g < s.n_gemm; ++g)
    if (s.gemm[g].xent_labels) prog.xent_g = g;
  prog.bar = bar_words;
  prog.wait_ns = wait_ns;
  prog.err = device_error_word();
  if (!prog.err) return MLP_ERR_CUDA;
  // a clean barrier count for this launch, even after an abandoned one
  if (cudaMemsetAsync(bar_words, 0, sizeof(unsigned), st) != cudaSuccess) return MLP_ERR_CUDA;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::SMEM + STEP_SGD_BYTES;  // epilogue staging and SGD state
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: the grid barrier needs it
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // recorded shape: steps, GEMM flops per step (2 M N K summed), GEMMs
  long long flops = 0;
  for (int g = 0; g < s.n_gemm; ++g)
    flops += 2ll * s.gemm[g].M * s.gemm[g].N * s.gemm[g].K;
  LaunchScope ls("step_program", st, s.n_steps, flops, s.n_gemm);
  const cudaError_t e =
      h16 ? cudaLaunchKernelEx(&cfg, tc_step_kernel<STEP_BN, STEP_STAGES, 1>, prog)
          : cudaLaunchKernelEx(&cfg, tc_step_kernel<STEP_BN, STEP_STAGES, 0>, prog);
  if (e != cudaSuccess) return MLP_ERR_CUDA;
  return launch_status();
}

size_t gemm_tc_splitk_bytes(int M, int N, int K) {
  const GemmPlan pl = gemm_plan(M, N, K, false);
  if (pl.splits <= 1) return 0;
  return (size_t)pl.splits * M * ((N + 3) / 4 * 4) * sizeof(float);
}

// The tile kernel for a planned GEMM, instantiated for its 16-bit format.
template <int H16>
mlp_status launch_tiles(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                        const TcParams& p, bool pair, int BN, cudaStream_t st) {
  if (pair) return launch_pair<6, H16>(ta, tb, tc, p, st);
  // short, narrow problems (the 784-256-10 step) need few stages
  if (BN == 64 && p.k_blocks <= 16) return launch_bn<64, 4, H16>(ta, tb, tc, p, st);
  switch (BN) {
    case 64: return launch_bn<64, 8, H16>(ta, tb, tc, p, st);
    case 128: return launch_bn<128, 6, H16>(ta, tb, tc, p, st);
    default: return launch_bn<256, 4, H16>(ta, tb, tc, p, st);
  }
}

mlp_status launch_gemm_tc(const GemmArgs& g, unsigned long long wait_ns, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0) return MLP_OK;
  if (g.K <= 0) {
    if (g.xent_labels || g.sgd_w) return MLP_ERR_UNSUPPORTED_SHAPE;
    return launch_gemm_simt(g, 1, st);
  }

  const bool fused = g.xent_labels || g.sgd_w;
  GemmPlan pl = gemm_plan(g.M, g.N, g.K, fused);
  if (pl.splits > 1 && !(g.ws && g.ws_bytes >= gemm_tc_splitk_bytes(g.M, g.N, g.K) &&
                         aligned16(g.ws))) {
    // no workspace for partial sums: one pass over K (single-CTA tiles when
    // the pair grid would be too small)
    pl.splits = 1;
    pl.kb_per_split = (g.K + BK - 1) / BK;
    if (((g.M + 255) / 256) * ((g.N + BN2 - 1) / BN2) < 48) pl.pair = false;
  }
  const int splits = pl.splits, kb_per_split = pl.kb_per_split;

  const int tiles_m = pl.pair ? (g.M + 255) / 256 : (g.M + BM - 1) / BM;
  // Widest tile that still gives every SM work; narrower tiles for small N.
  int BN = 256;
  const int sms = num_sms();
  auto tiles_for = [&](int bn) { return tiles_m * ((g.N + bn - 1) / bn); };
  if (pl.pair || splits > 1) BN = 256;
  else if (g.N <= 64) BN = 64;
  else if (g.N <= 128) BN = 128;
  else if (tiles_for(256) < sms) BN = tiles_for(128) < sms ? 64 : 128;
  if (!pl.pair && splits == 1 && BN == 128 && tiles_for(128) < sms / 2 && g.N > 64) BN = 64;

  CUtensorMap ta, tb;
  TcParams p;
  MLP_CHECK(prepare_tc(g, tiles_m, BN, splits, kb_per_split, pl.pair ? 128 : BN, wait_ns, &p, &ta,
                       &tb));

  // Output through TMA stores when the output is large (for small outputs the
  // staging round trip costs more latency than it saves), rows are 16-byte
  // aligned and no fused epilogue writes extra tensors.
  CUtensorMap tc;
  memset(&tc, 0, sizeof(tc));
  const int esz = g.c_bf16 ? 2 : 4;
  p.tma_store = 0;
  if (!p.xent_labels && !p.sgd_w && splits == 1 && (long long)g.M * g.N >= (1ll << 20) &&
      ((long long)g.ldc * esz) % 16 == 0 && aligned16(g.C)) {
    if (!encode_tmap_out_2d(&tc, g.C, g.c_bf16 ? 0 : 1, g.N, g.M,
                            (unsigned long long)g.ldc * esz, 32, 32))
      return MLP_ERR_CUDA;
    p.tma_store = 1;
  }
  return p.f16 ? launch_tiles<1>(ta, tb, tc, p, pl.pair, BN, st)
               : launch_tiles<0>(ta, tb, tc, p, pl.pair, BN, st);
}

// QKV projection with the fused attention-preprocessing epilogue: CTA-pair
// 256 x 256 tiles (each a whole number of 64-column heads), one pass over K,
// bf16 operands and output.
mlp_status launch_attn_prep_gemm(const GemmArgs& g, const float* rstd, const float* q_gain,
                                 int n_q, int n_kv, int rope_dims, int seq_len, float eps,
                                 float theta, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0) return MLP_OK;
  if (g.K <= 0 || !g.c_bf16 || g.f16 || g.bias || g.mask || g.act != MLP_ACT_NONE ||
      (rope_dims != 16 && rope_dims != 32 && rope_dims != 64) || g.N != (n_q + 2 * n_kv) * 64)
    return MLP_ERR_UNSUPPORTED_SHAPE;
  CUtensorMap ta, tb, tc;
  TcParams p;
  const unsigned long long wait_ns = wait_limit_ns();
  MLP_CHECK(prepare_tc(g, (g.M + 255) / 256, BN2, 1, (g.K + BK - 1) / BK, 128, wait_ns, &p, &ta,
                       &tb));
  memset(&tc, 0, sizeof(tc));
  p.tma_store = 0;
  if ((long long)g.M * g.N >= (1ll << 20) && ((long long)g.ldc * 2) % 16 == 0 && aligned16(g.C)) {
    // one head (64 columns) per store: 32 x 64 boxes, 128-byte swizzle
    if (!encode_tmap_bf16_2d(&tc, g.C, g.N, g.M, (unsigned long long)g.ldc * 2, 64, 32))
      return MLP_ERR_CUDA;
    p.tma_store = 1;
  }
  AttnEpi ae{};
  ae.rstd = rstd;
  ae.q_gain = q_gain;
  ae.n_q = n_q;
  ae.n_qk = n_q + n_kv;
  ae.seq_len = seq_len;
  ae.eps = eps;
  ae.theta = theta;
  // K up to 512: the weights stay resident and only the token rows stream
  if (p.k_blocks <= kBResBlocks) {
    switch (rope_dims) {
      case 16: return launch_pair<4, 0, 16, true>(ta, tb, tc, p, st, ae);
      case 32: return launch_pair<4, 0, 32, true>(ta, tb, tc, p, st, ae);
      default: return launch_pair<4, 0, 64, true>(ta, tb, tc, p, st, ae);
    }
  }
  switch (rope_dims) {
    case 16: return launch_pair<5, 0, 16>(ta, tb, tc, p, st, ae);
    case 32: return launch_pair<5, 0, 32>(ta, tb, tc, p, st, ae);
    default: return launch_pair<5, 0, 64>(ta, tb, tc, p, st, ae);
  }
}

}  // namespace mlp
