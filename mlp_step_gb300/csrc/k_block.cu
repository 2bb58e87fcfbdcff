// Transformer MLP block kernels for sm_103a ("Full-Depth MLP Megakernel +
// Fused Attention Preprocessing", "What Worked": RMSNorm -> gate projection ->
// LeakyReLU^2 -> down projection -> residual, the wide intermediate never
// written to memory).
//
// Forward (block_fwd_kernel): one CTA pair (a 2-CTA cluster) per 128-token
// tile, the gate computed transposed (hidden units on tensor-memory lanes,
// tokens on columns) by tcgen05.mma.cta_group::2, so each CTA keeps only its
// 64 tokens of x in shared memory for the whole tile; the activation epilogue
// writes each token's bf16 activations into the down MMA's operand slot of the
// CTA that supplies that token (one of the two by distributed shared memory),
// and the down projection accumulates Y^T in tensor memory.  No FLOP is
// recomputed and the intermediate stays on chip (the page's design kept it in
// registers and lost to one large library GEMM; here it lives in tensor memory
// and shared memory and is fed to the tensor cores directly).  Details at the
// kernel.
//
// RMSNorm with gain 1 is folded into the epilogue: u = r (x W_gate) with
// r = 1 / sqrt(mean(x^2) + eps) per token, so the gate GEMM reads x as is.
//
// Backward (block_bwd_act_kernel): per 256-token x 256-hidden tile, two MMA
// accumulators U = x W_gate[:, c] and DA = dy W_down[c, :]^T over K = 512,
// computed one after the other by a CTA pair with tcgen05.mma.cta_group::2
// (each CTA stages its own 128 token rows of x and dy and half of the tile's
// weight columns); the epilogue converts each accumulator while the other is
// being computed and writes a = f(r U) and r du = DA r f'(r U) in bf16 for
// the weight-gradient GEMMs, through TMA bulk stores.  rmsnorm_bwd_kernel
// finishes dx from dn' = (r du) W_gate^T.
#include "kernels.cuh"
#include "ptx.cuh"
#include "trace.cuh"

namespace mlp {

namespace {

constexpr int TM = 128;                 // tokens per tile (forward: per CTA pair)
constexpr int DM = 512;                 // model width

__device__ __forceinline__ float lrelu_sq(float u, float slope) {
  const float t = u > 0.f ? u : slope * u;
  return t * t;
}

__device__ __forceinline__ float lrelu_sq_grad(float u, float slope) {
  return u > 0.f ? 2.f * u : 2.f * slope * slope * u;
}

__device__ __forceinline__ float sumsq_bf16x8(const uint4& v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    s += f.x * f.x;
    s += f.y * f.y;
  }
  return s;
}

// ------------------------------------------------------------------ forward

// Forward megakernel on CTA pairs with the gate computed transposed.  A pair
// (2-CTA cluster) owns a tile of 128 tokens; CTA r supplies tokens
// [64 r, 64 r + 64) of it as MMA operands and holds those tokens of x in
// shared memory for the whole tile (read from memory once per tile).  For
// each 256-wide hidden chunk c:
//   gate:  G_c^T [256 hidden, 128 tokens] = W_gate[:, c]^T x^T   (K = 512)
//          one tcgen05.mma.cta_group::2 of M = 256, N = 128: CTA r stages
//          hidden rows [128 r, 128 r + 128) of the chunk (W_gate read as an
//          M-major operand) and receives them in its tensor memory, lanes =
//          hidden units, columns = the tile's 128 tokens;
//   act:   eight epilogue warps per CTA read G_c^T, form a = f(r_t g) in fp32
//          (RMSNorm's row scale r_t of token t, LeakyReLU^2), round to bf16
//          and write each token's activations where the down MMA reads them:
//          tokens [0, 64) into CTA 0's slot, [64, 128) into CTA 1's (one of
//          the two by distributed shared memory);
//   down:  Y^T [512 out, 128 tokens] += W_down[c, :]^T A_c^T     (K = 256)
//          two M = 256 pair MMAs (output columns [0, 256) and [256, 512)),
//          B = the activation slot (MN-major, tokens contiguous).
// Tensor memory per CTA: Y^T (its 256 output columns x 128 tokens, 256
// columns) and two 128-column gate accumulators, so the gate of chunk c + 1
// runs while the epilogue converts chunk c; two activation slots let the down
// MMAs of chunk c run while chunk c + 1's activations are written.  MMA order
// per tile: G0 G1 D0 G2 D1 ... G_{n-1} D_{n-2} D_{n-1}.  Four output warps
// per CTA compute the next tile's row scales from the resident x, then drain
// Y^T (+ x, bf16) while the next tile's first two gates run.
// The intermediate never leaves tensor and shared memory.
constexpr int F2_TOK = 64;                   // tokens per CTA per tile
constexpr int F2_HC = 256;                   // hidden per chunk (pair M)
constexpr int F2_X_BYTES = F2_TOK * DM * 2;  // 64 KiB: 8 k-blocks of [64 tokens][128 B]
constexpr int F2_SLOT_BYTES = F2_HC * F2_TOK * 2;  // 32 KiB: [256 hidden][64 tokens] bf16
constexpr int F2_STAGES = 3;
constexpr int F2_STAGE_BYTES = 32768;
constexpr int F2_X = 0;
constexpr int F2_SLOTS = F2_X + F2_X_BYTES;
constexpr int F2_STG = F2_SLOTS + 2 * F2_SLOT_BYTES;
constexpr int F2_RBUF = F2_STG + F2_STAGES * F2_STAGE_BYTES;  // float [2][128]
constexpr int F2_BARS = F2_RBUF + 2 * TM * 4;
constexpr int F2_SMEM = 1024 + F2_BARS + 256;
constexpr int F2_THREADS = 448;  // producer, MMA, 4 output warps, 8 epilogue warps
static_assert(F2_SMEM <= 232448, "forward kernel shared memory");

struct Fwd2Params {
  int T, n_chunks, tiles;
  float eps, slope;
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  float* rstd;
  unsigned long long wait_ns;
  int* err;
};

// MMA / weight-stream order of one tile: op i -> (is_down, chunk).
__device__ __forceinline__ void f2_op(int i, int n, bool& down, int& c) {
  // G0, then (G_j, D_{j-1}) for j = 1 .. n-1, then D_{n-1}
  if (i == 0) { down = false; c = 0; return; }
  if (i == 2 * n - 1) { down = true; c = n - 1; return; }
  const int j = (i + 1) >> 1;
  down = (i & 1) == 0;
  c = down ? j - 1 : j;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(F2_THREADS, 1)
    block_fwd_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmWg,
                     const __grid_constant__ CUtensorMap tmWd, const Fwd2Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* xs = smem + F2_X;
  uint8_t* slots = smem + F2_SLOTS;
  uint8_t* stages = smem + F2_STG;
  float* rbuf = reinterpret_cast<float*>(smem + F2_RBUF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + F2_BARS);
  uint64_t* empty = full + F2_STAGES;
  uint64_t* gfull = empty + F2_STAGES;   // [2] gate accumulator ready (multicast commit)
  uint64_t* gempty = gfull + 2;          // [2] drained (leader: 16 warp arrivals)
  uint64_t* afull = gempty + 2;          // [2] slot written (leader: 512 thread arrivals)
  uint64_t* aempty = afull + 2;          // [2] slot consumed (multicast commit)
  uint64_t* xfull = aempty + 2;          // this CTA's x landed (tx bytes)
  uint64_t* xempty = xfull + 1;          // last gate of the tile done (multicast commit)
  uint64_t* rready = xempty + 1;         // [2] row scales of a tile in rbuf (256 arrivals)
  uint64_t* yfull = rready + 2;          // Y^T complete (multicast commit)
  uint64_t* yempty = yfull + 1;          // Y^T drained (leader: 8 warp arrivals)
  uint64_t* done = yempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int cluster = blockIdx.x >> 1;
  const int n_clusters = gridDim.x >> 1;
  const int n = p.n_chunks;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < F2_STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&gfull[b], 1);
      ptx::mbar_init(&gempty[b], 16);
      ptx::mbar_init(&afull[b], 512);
      ptx::mbar_init(&aempty[b], 1);
      ptx::mbar_init(&rready[b], 256);
    }
    ptx::mbar_init(xfull, 1);
    ptx::mbar_init(xempty, 1);
    ptx::mbar_init(yfull, 1);
    ptx::mbar_init(yempty, 8);
    ptx::mbar_init(done, 1);
    *s_abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tmX);
    ptx::prefetch_tensormap(&tmWg);
    ptx::prefetch_tensormap(&tmWd);
  }
  if (warp == 1) ptx::tmem_alloc_pair(tmem_slot, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  ptx::tc_fence_after();
  // Y^T: columns [0, 128) output half 0, [128, 256) half 1; gate buffers at
  // 256 and 384
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();

  int last_parity[F2_STAGES];
  int x_parity = -1;

  if (warp == 0) {
    // ---------------------------------------------------------------- weights producer
    if (lane == 0) {
      for (int s = 0; s < F2_STAGES; ++s) last_parity[s] = -1;
      const uint32_t full0 = ptx::mapa_shared(ptx::smem_u32(full), 0);  // the leader's full[]
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = cluster; t < p.tiles && ok && !*s_abort; t += n_clusters) {
        for (int i = 0; i < 2 * n && ok; ++i) {
          bool down;
          int c;
          f2_op(i, n, down, c);
          for (int q = 0; q < 4; ++q) {
            if (!ptx::mbar_wait_cluster_bounded(&empty[stage], phase ^ 1, p.wait_ns, p.err,
                                                DEVERR_TIMEOUT_PRODUCER)) {
              *s_abort = 1;
              ok = false;
              break;
            }
            if (rank == 0) {
              ptx::mbar_arrive_expect_tx(&full[stage], 2 * F2_STAGE_BYTES);
              last_parity[stage] = (int)phase;
            }
            const uint32_t bar = full0 + (uint32_t)stage * 8u;
            uint8_t* st = stages + stage * F2_STAGE_BYTES;
            if (!down) {
              // W_gate^T rows (hidden) [c*256 + 128 r, +128) x d [128 q, +128): two
              // 64-hidden boxes of 128 d rows
              const int h0 = c * F2_HC + (int)rank * 128;
              ptx::tma_load_2d_pair(st, &tmWg, bar, h0, q * 128);
              ptx::tma_load_2d_pair(st + 16384, &tmWg, bar, h0 + 64, q * 128);
            } else {
              // W_down^T rows (output columns) of both halves x hidden [c*256 + 64 q, +64)
              const int k0 = c * F2_HC + q * 64;
#pragma unroll
              for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int b = 0; b < 2; ++b)
                  ptx::tma_load_2d_pair(st + hh * 16384 + b * 8192, &tmWd, bar,
                                        hh * 256 + (int)rank * 128 + b * 64, k0);
            }
            if (++stage == F2_STAGES) { stage = 0; phase ^= 1; }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      const uint32_t idesc_g = ptx::idesc_bf16_f32(2 * TM, TM, 1, 0);  // A M-major, B K-major
      const uint32_t idesc_d = ptx::idesc_bf16_f32(2 * TM, TM, 1, 1);  // A M-major, B MN-major
      const uint32_t xs_a = ptx::smem_u32(xs);
      const uint32_t slot_a = ptx::smem_u32(slots);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = cluster; t < p.tiles && ok && !*s_abort; t += n_clusters, ++it) {
        // both CTAs' x for this tile have landed (the row-scale warps arrive
        // after seeing their own x)
        if (!ptx::mbar_wait_cluster_bounded(&rready[it & 1], (it >> 1) & 1, p.wait_ns, p.err,
                                            DEVERR_TIMEOUT_MMA)) { ok = false; break; }
        for (int i = 0; i < 2 * n && ok; ++i) {
          bool down;
          int c;
          f2_op(i, n, down, c);
          const uint32_t g = (uint32_t)(it * n + c);  // running chunk index
          const int b = (int)(g & 1);
          if (!down) {
            if (!ptx::mbar_wait_cluster_bounded(&gempty[b], ((g >> 1) & 1) ^ 1, p.wait_ns, p.err,
                                                DEVERR_TIMEOUT_MMA)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t d = tmem + 256 + (uint32_t)b * 128;
            for (int q = 0; q < 4; ++q) {
              if (!ptx::mbar_wait_bounded(&full[stage], phase, p.wait_ns, p.err,
                                          DEVERR_TIMEOUT_MMA)) { ok = false; break; }
              ptx::tc_fence_after();
              const uint32_t sa = ptx::smem_u32(stages + stage * F2_STAGE_BYTES);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const int kk = q * 128 + k * 16;  // d index of this K step
                const uint64_t ad = ptx::sw128_desc(sa + k * 2048, 16384, 1024);
                const uint64_t bd =
                    ptx::sw128_desc(xs_a + (kk >> 6) * 8192 + (kk & 63) * 2, 16, 1024);
                ptx::mma_bf16_pair(d, ad, bd, idesc_g, (q > 0 || k > 0) ? 1u : 0u);
              }
              ptx::mma_commit_pair_multicast(&empty[stage], 3);
              if (++stage == F2_STAGES) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            ptx::mma_commit_pair_multicast(&gfull[b], 3);
            if (c == n - 1) ptx::mma_commit_pair_multicast(xempty, 3);
          } else {
            if (c == 0) {
              if (!ptx::mbar_wait_cluster_bounded(yempty, (it & 1) ^ 1, p.wait_ns, p.err,
                                                  DEVERR_TIMEOUT_MMA)) { ok = false; break; }
            }
            if (!ptx::mbar_wait_cluster_bounded(&afull[b], (g >> 1) & 1, p.wait_ns, p.err,
                                                DEVERR_TIMEOUT_PEER)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t sl = slot_a + (uint32_t)b * F2_SLOT_BYTES;
            for (int q = 0; q < 4; ++q) {
              if (!ptx::mbar_wait_bounded(&full[stage], phase, p.wait_ns, p.err,
                                          DEVERR_TIMEOUT_MMA)) { ok = false; break; }
              ptx::tc_fence_after();
              const uint32_t sa = ptx::smem_u32(stages + stage * F2_STAGE_BYTES);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t bd = ptx::sw128_desc(sl + (q * 64 + k * 16) * 128, 8192, 1024);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  const uint64_t ad = ptx::sw128_desc(sa + hh * 16384 + k * 2048, 8192, 1024);
                  ptx::mma_bf16_pair(tmem + (uint32_t)hh * 128, ad, bd, idesc_d,
                                     (c > 0 || q > 0 || k > 0) ? 1u : 0u);
                }
              }
              ptx::mma_commit_pair_multicast(&empty[stage], 3);
              if (++stage == F2_STAGES) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            ptx::mma_commit_pair_multicast(&aempty[b], 3);
            if (c == n - 1) ptx::mma_commit_pair_multicast(yfull, 3);
          }
        }
      }
      if (!ok) *s_abort = 1;
      ptx::mma_commit_pair_multicast(done, 1);
      ptx::mbar_wait_bounded(done, 0, p.wait_ns, p.err, DEVERR_TIMEOUT_TEARDOWN);
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------------- x, row scales, output
    // Thread (quarter q, lane l) owns tensor-memory lane 32 q + l: output
    // column 256 hh + 128 rank + 32 q + l of half hh.
    const int quarter = warp & 3;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t yempty0 = ptx::mapa_shared(ptx::smem_u32(yempty), 0);
    const uint32_t rbuf_peer = ptx::mapa_shared(ptx::smem_u32(rbuf), peer);
    const uint32_t rready_peer = ptx::mapa_shared(ptx::smem_u32(rready), peer);
    // row scales: two threads per token, each summing half of the row
    const int tok = (warp - 2) * 16 + (lane >> 1);
    const int rhalf = lane & 1;
    bool ok = true;
    int it = 0;
    int t_prev = -1;
    auto drain = [&](int tp, int itp) -> bool {
      if (!ptx::mbar_wait_bounded(yfull, itp & 1, p.wait_ns, p.err, DEVERR_TIMEOUT_EPILOGUE))
        return false;
      ptx::tc_fence_after();
      const int odd = lane & 1;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        // this lane's pair of output columns (even lane: o, o+1; odd: o-1, o)
        const int col = hh * 256 + (int)rank * 128 + quarter * 32 + (lane & ~1);
#pragma unroll 1
        for (int tb = 0; tb < TM / 32; ++tb) {
          uint32_t v[32];
          __syncwarp();
          ptx::tmem_ld_32x32b_x32(tmem + lane_off + (uint32_t)(hh * 128 + tb * 32), v);
          ptx::tmem_ld_wait();
          if (hh == 1 && tb == TM / 32 - 1) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (rank == 0) ptx::mbar_arrive(yempty);
              else ptx::mbar_arrive_remote(yempty0);
            }
          }
          // token pairs (j, j+1): even lanes take token j, odd lanes j + 1
          uint32_t xv[16];
          const int m0 = tp * TM + tb * 32 + odd;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int m = m0 + 2 * jj;
            xv[jj] = m < p.T ? __ldg(reinterpret_cast<const unsigned int*>(
                                   p.x + (size_t)m * DM + col))
                             : 0u;
          }
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const float send = __uint_as_float(odd ? v[2 * jj] : v[2 * jj + 1]);
            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
            const float lo = odd ? recv : __uint_as_float(v[2 * jj]);
            const float hi = odd ? __uint_as_float(v[2 * jj + 1]) : recv;
            const int m = m0 + 2 * jj;
            if (m < p.T) {
              const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xv[jj]));
              *reinterpret_cast<unsigned int*>(p.y + (size_t)m * DM + col) =
                  pack_bf16x2(lo + xf.x, hi + xf.y);
            }
          }
        }
      }
      return true;
    };
    for (int t = cluster; t < p.tiles && ok; t += n_clusters, ++it) {
      if (*s_abort) { ok = false; break; }
      // this CTA's 64 tokens of x, once the last gate of the tile before has run
      if (warp == 2 && lane == 0) {
        if (it > 0 && !ptx::mbar_wait_bounded(xempty, (it - 1) & 1, p.wait_ns, p.err,
                                               DEVERR_TIMEOUT_EPILOGUE)) {
          *s_abort = 1;
        } else {
          ptx::mbar_arrive_expect_tx(xfull, (uint32_t)F2_X_BYTES);
          x_parity = it & 1;
#pragma unroll
          for (int kb = 0; kb < DM / 64; ++kb)
            ptx::tma_load_2d(xs + kb * 8192, &tmX, xfull, kb * 64, t * TM + (int)rank * F2_TOK);
        }
      }
      __syncwarp();
      if (!ptx::mbar_wait_bounded(xfull, it & 1, p.wait_ns, p.err, DEVERR_TIMEOUT_EPILOGUE)) {
        ok = false;
        break;
      }
      // row scale of token `tok`: sum of squares over this thread's four
      // k-blocks, 16-byte chunks read in swizzled order (conflict-free)
      float ss = 0.f;
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) {
        const uint8_t* row = xs + (rhalf * 4 + kb) * 8192 + tok * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          ss += sumsq_bf16x8(*reinterpret_cast<const uint4*>(row + ((j ^ (tok & 7)) << 4)));
      }
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      const int m = t * TM + (int)rank * F2_TOK + tok;
      const float r = m < p.T ? 1.0f / sqrtf(ss / (float)DM + p.eps) : 0.f;
      const int buf = it & 1;
      if (rhalf == 0) {
        const int idx = buf * TM + (int)rank * F2_TOK + tok;
        rbuf[idx] = r;
        ptx::st_cluster_f32(rbuf_peer + (uint32_t)idx * 4u, r);
        if (p.rstd && m < p.T) p.rstd[m] = r;
      }
      ptx::mbar_arrive_cluster_local(&rready[buf]);
      ptx::mbar_arrive_remote(rready_peer + (uint32_t)buf * 8u);
      // output of the tile before, while this tile's first gates run
      if (t_prev >= 0 && !drain(t_prev, it - 1)) { ok = false; break; }
      t_prev = t;
    }
    if (ok && t_prev >= 0 && !*s_abort && !drain(t_prev, it - 1)) ok = false;
    if (!ok) *s_abort = 1;
  } else {
    // ---------------------------------------------------------------- gate epilogue
    // Warps 6-13: tensor-memory lane quarter warp % 4 (hidden units), token
    // half th (columns [64 th, 64 th + 64)); the activations of those tokens
    // go to CTA th's slot.
    const int quarter = warp & 3;
    const int th = (warp - 6) >> 2;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t gempty0 = ptx::mapa_shared(ptx::smem_u32(gempty), 0);
    const uint32_t afull0 = ptx::mapa_shared(ptx::smem_u32(afull), 0);
    const int k = (int)rank * 128 + quarter * 32 + lane;  // hidden row within the chunk
    const uint32_t dst_slots = ptx::mapa_shared(ptx::smem_u32(slots), (uint32_t)th);
    bool ok = true;
    int it = 0;
    for (int t = cluster; t < p.tiles && ok; t += n_clusters, ++it) {
      const float* rt = rbuf + (it & 1) * TM + th * F2_TOK;
      for (int c = 0; c < n && ok; ++c) {
        if (*s_abort) { ok = false; break; }
        const uint32_t g = (uint32_t)(it * n + c);
        const int b = (int)(g & 1);
        if (!ptx::mbar_wait_bounded(&gfull[b], (g >> 1) & 1, p.wait_ns, p.err,
                                    DEVERR_TIMEOUT_EPILOGUE)) { ok = false; break; }
        ptx::tc_fence_after();
        uint32_t v[64];
        __syncwarp();
        ptx::tmem_ld_32x32b_x32(tmem + lane_off + 256 + (uint32_t)(b * 128 + th * 64),
                                *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        ptx::tmem_ld_32x32b_x32(tmem + lane_off + 256 + (uint32_t)(b * 128 + th * 64 + 32),
                                *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        ptx::tmem_ld_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) ptx::mbar_arrive(&gempty[b]);
          else ptx::mbar_arrive_remote(gempty0 + (uint32_t)b * 8u);
        }
        if (c == 0 && !ptx::mbar_wait_cluster_bounded(&rready[it & 1], (it >> 1) & 1, p.wait_ns,
                                                      p.err, DEVERR_TIMEOUT_EPILOGUE)) {
          ok = false;
          break;
        }
        if (!ptx::mbar_wait_bounded(&aempty[b], ((g >> 1) & 1) ^ 1, p.wait_ns, p.err,
                                    DEVERR_TIMEOUT_EPILOGUE)) { ok = false; break; }
        const uint32_t row = dst_slots + (uint32_t)(b * F2_SLOT_BYTES + k * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 r0 = *reinterpret_cast<const float4*>(rt + 8 * j);
          const float4 r1 = *reinterpret_cast<const float4*>(rt + 8 * j + 4);
          const float* u = reinterpret_cast<const float*>(&v[8 * j]);
          uint4 o;
          o.x = pack_bf16x2(lrelu_sq(u[0] * r0.x, p.slope), lrelu_sq(u[1] * r0.y, p.slope));
          o.y = pack_bf16x2(lrelu_sq(u[2] * r0.z, p.slope), lrelu_sq(u[3] * r0.w, p.slope));
          o.z = pack_bf16x2(lrelu_sq(u[4] * r1.x, p.slope), lrelu_sq(u[5] * r1.y, p.slope));
          o.w = pack_bf16x2(lrelu_sq(u[6] * r1.z, p.slope), lrelu_sq(u[7] * r1.w, p.slope));
          ptx::st_cluster_v4(row + (uint32_t)((j ^ (k & 7)) << 4), o);
        }
        ptx::fence_proxy_async_cluster();
        if (rank == 0) ptx::mbar_arrive_cluster_local(&afull[b]);
        else ptx::mbar_arrive_remote(afull0 + (uint32_t)b * 8u);
      }
    }
    if (!ok) *s_abort = 1;
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (*s_abort && warp == 0 && lane == 0) {
    for (int s = 0; s < F2_STAGES; ++s)
      if (last_parity[s] >= 0)
        ptx::mbar_wait_bounded(&full[s], (uint32_t)last_parity[s], p.wait_ns, p.err,
                               DEVERR_TIMEOUT_TEARDOWN);
  }
  if (*s_abort && warp == 2 && lane == 0 && x_parity >= 0)
    ptx::mbar_wait_bounded(xfull, (uint32_t)x_parity, p.wait_ns, p.err, DEVERR_TIMEOUT_TEARDOWN);
  __syncwarp();
  __syncthreads();
  // neither CTA frees its tensor memory or leaves while the pair's MMAs,
  // copies or signals may still reach it
  ptx::cluster_sync();
  if (warp == 1) {
    __syncwarp();
    ptx::tmem_dealloc_pair(tmem, 512);
  }
}

// ------------------------------------------------------------------ backward

// Each pair tile covers 256 tokens x BH = 256 hidden columns and runs as two
// halves: U = x W_gate[:, tile] (K = 512) into tensor-memory columns
// [0, 256), then DA = dy W_down[tile, :]^T into columns [256, 512).  Stage
// one of the epilogue converts U (writes a = f(r U), keeps g = r f'(r U) as
// packed bf16 in registers) while the MMA computes DA; stage two forms
// r du = DA g while the MMA computes the next tile's U.  So the MMA never
// waits for a whole-tile epilogue, and every x / dy k-block feeds 256 hidden
// columns (the kernel is bound by how fast TMA fills one SM's shared memory
// from L2, ~89 GB/s per SM on this part).
//
// A stage holds one half's operands for one 64-wide k-block: x or dy rows
// (16 KiB) and this CTA's 128 W_gate columns (two 8 KiB boxes) or 128 W_down
// rows (16 KiB).
constexpr int BH = 256;
constexpr int B_STAGES = 6;
constexpr int B_A = 0, B_B = 16384;
constexpr int B_STAGE_BYTES = 32768;
constexpr int B_BAR_BYTES = 1024;
constexpr int B_THREADS = 320;        // producer, MMA, 8 epilogue warps
constexpr int B_STG_BYTES = 8 * 4096;  // per epilogue warp: 2 buffers x 2 KiB
constexpr int B_SMEM = 1024 + B_STAGES * B_STAGE_BYTES + B_BAR_BYTES + B_STG_BYTES;
static_assert(B_SMEM <= 232448, "backward kernel shared memory");

struct BwdParams {
  int T, hidden, pairs_m, tiles_h, num_tiles;
  float slope;
  const float* rstd;
  unsigned long long wait_ns;
  int* err;
};

// Tile t covers token rows [256 pm, 256 pm + 256) and hidden columns
// [256 th, 256 th + 256).  Four token pairs at a time sweep all hidden
// chunks (the last group may be shorter), so pairs running together share
// x / dy rows and weight columns in L2.
__device__ __forceinline__ void bwd_tile(int t, int pairs_m, int tiles_h, int& pm, int& th) {
  constexpr int G = 4;
  const int group = t / (G * tiles_h);
  const int first = group * G;
  const int gm = min(pairs_m - first, G);
  const int r = t - group * G * tiles_h;
  pm = first + r % gm;
  th = r / gm;
}

// Row `lane` of a warp's 32 x 32 bf16 staging box in the 64-byte-swizzled
// layout of the output tensor maps: 16-byte chunk q at q ^ ((lane >> 1) & 3).
__device__ __forceinline__ void stage_row_bf16(uint8_t* box, int lane, const uint32_t (&pk)[16]) {
  uint8_t* row = box + lane * 64;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(row + ((q ^ ((lane >> 1) & 3)) << 4)) =
        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
}

// One epilogue warp's 32 x 32 bf16 box through its double-buffered staging
// area and a TMA store (rows past the last token are clipped by the map).
__device__ __forceinline__ void store_box_bf16(const CUtensorMap* map, uint8_t* wstg,
                                               int& stg_count, int lane,
                                               const uint32_t (&pk)[16], int col, int row) {
  uint8_t* box = wstg + (stg_count & 1) * 2048;
  if (stg_count >= 2) {
    if (lane == 0) ptx::bulk_wait_group_read<1>();
    __syncwarp();
  }
  stage_row_bf16(box, lane, pk);
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    ptx::tma_store_2d(map, box, col, row);
    ptx::bulk_commit_group();
  }
  ++stg_count;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(B_THREADS, 1)
    block_bwd_act_kernel(const __grid_constant__ CUtensorMap tmX,
                         const __grid_constant__ CUtensorMap tmWg,
                         const __grid_constant__ CUtensorMap tmDy,
                         const __grid_constant__ CUtensorMap tmWd,
                         const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmDu, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + B_STAGES * B_STAGE_BYTES);
  uint8_t* stg = stages + B_STAGES * B_STAGE_BYTES + B_BAR_BYTES;
  uint64_t* empty = full + B_STAGES;
  uint64_t* tfull = empty + B_STAGES;  // [half]: accumulator ready
  uint64_t* tempty = tfull + 2;        // [half]: accumulator read out
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < B_STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int h = 0; h < 2; ++h) {
      ptx::mbar_init(&tfull[h], 1);
      ptx::mbar_init(&tempty[h], 16);  // the pair's sixteen epilogue warps
    }
    ptx::mbar_init(done, 1);
    *s_abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tmX);
    ptx::prefetch_tensormap(&tmWg);
    ptx::prefetch_tensormap(&tmDy);
    ptx::prefetch_tensormap(&tmWd);
    ptx::prefetch_tensormap(&tmA);
    ptx::prefetch_tensormap(&tmDu);
  }
  if (warp == 1) ptx::tmem_alloc_pair(tmem_slot, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // U at column 0, DA at column BH
  pdl_wait();
  pdl_launch_dependents();
  int last_parity[B_STAGES];

  if (warp == 0) {
    if (lane == 0) {
      for (int s = 0; s < B_STAGES; ++s) last_parity[s] = -1;
      const uint32_t full0 = ptx::mapa_shared(ptx::smem_u32(full), 0);  // the even CTA's full[]
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = pair; t < p.num_tiles && ok && !*s_abort; t += n_pairs) {
        int pm, th;
        bwd_tile(t, p.pairs_m, p.tiles_h, pm, th);
        const int m0 = pm * 2 * TM + (int)rank * TM;
        const int h0 = th * BH + (int)rank * (BH / 2);
        for (int half = 0; half < 2 && ok; ++half) {
          for (int kb = 0; kb < DM / 64; ++kb) {
            if (!ptx::mbar_wait_cluster_bounded(&empty[stage], phase ^ 1, p.wait_ns, p.err,
                                                DEVERR_TIMEOUT_PRODUCER)) {
              *s_abort = 1;
              ok = false;
              break;
            }
            if (rank == 0) {
              ptx::mbar_arrive_expect_tx(&full[stage], 2 * B_STAGE_BYTES);
              last_parity[stage] = (int)phase;
            }
            const uint32_t bar = full0 + (uint32_t)stage * 8u;
            uint8_t* st = stages + stage * B_STAGE_BYTES;
            if (half == 0) {
              ptx::tma_load_2d_pair(st + B_A, &tmX, bar, kb * 64, m0);
              ptx::tma_load_2d_pair(st + B_B, &tmWg, bar, h0, kb * 64);
              ptx::tma_load_2d_pair(st + B_B + 8192, &tmWg, bar, h0 + 64, kb * 64);
            } else {
              ptx::tma_load_2d_pair(st + B_A, &tmDy, bar, kb * 64, m0);
              ptx::tma_load_2d_pair(st + B_B, &tmWd, bar, kb * 64, h0);
            }
            if (++stage == B_STAGES) { stage = 0; phase ^= 1; }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // half 0: B = W_gate columns (N-major); half 1: B = W_down rows (K-major)
      const uint32_t idesc[2] = {ptx::idesc_bf16_f32(2 * TM, BH, 0, 1),
                                 ptx::idesc_bf16_f32(2 * TM, BH, 0, 0)};
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = pair; t < p.num_tiles && ok && !*s_abort; t += n_pairs) {
        for (int half = 0; half < 2; ++half) {
          if (!ptx::mbar_wait_cluster_bounded(&tempty[half], acc_phase ^ 1, p.wait_ns, p.err,
                                              DEVERR_TIMEOUT_MMA)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(half * BH);
          for (int kb = 0; kb < DM / 64; ++kb) {
            if (!ptx::mbar_wait_bounded(&full[stage], phase, p.wait_ns, p.err,
                                        DEVERR_TIMEOUT_MMA)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t sb = ptx::smem_u32(stages + stage * B_STAGE_BYTES);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t bd = half == 0 ? ptx::sw128_desc(sb + B_B + k * 2048, 8192, 1024)
                                            : ptx::sw128_desc(sb + B_B + k * 32, 16, 1024);
              ptx::mma_bf16_pair(d, ptx::sw128_desc(sb + B_A + k * 32, 16, 1024), bd,
                                 idesc[half], (kb > 0 || k > 0) ? 1u : 0u);
            }
            ptx::mma_commit_pair_multicast(&empty[stage], 3);
            if (++stage == B_STAGES) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          ptx::mma_commit_pair_multicast(&tfull[half], 3);
        }
        acc_phase ^= 1;
      }
      if (!ok) *s_abort = 1;
      ptx::mma_commit_pair_multicast(done, 1);
      ptx::mbar_wait_bounded(done, 0, p.wait_ns, p.err, DEVERR_TIMEOUT_TEARDOWN);
    }
  } else {
    // Warps 2-9: TMEM lane quarter warp % 4, columns [c_half, c_half + 128)
    // of the tile.
    const int quarter = warp & 3;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int c_half = ((warp - 2) >> 2) * (BH / 2);
    const uint32_t tempty0 = ptx::mapa_shared(ptx::smem_u32(tempty), 0);
    uint8_t* wstg = stg + (warp - 2) * 4096;
    uint32_t acc_phase = 0;
    int stg_count = 0;
    bool ok = true;
    for (int t = pair; t < p.num_tiles && ok; t += n_pairs) {
      int pm, th;
      bwd_tile(t, p.pairs_m, p.tiles_h, pm, th);
      const int row0 = pm * 2 * TM + (int)rank * TM + quarter * 32;  // this warp's first row
      const int m = row0 + lane;
      const float r = m < p.T ? __ldg(p.rstd + m) : 0.f;
      const int col0 = th * BH + c_half;
      uint32_t g[BH / 4];  // r f'(r U) as packed bf16 pairs, 128 columns
      for (int half = 0; half < 2; ++half) {
        if (*s_abort) { ok = false; break; }
        if (!ptx::mbar_wait_cluster_bounded(&tfull[half], acc_phase, p.wait_ns, p.err,
                                            DEVERR_TIMEOUT_EPILOGUE)) {
          *s_abort = 1;
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < BH / 64; ++cc) {
          uint32_t v[32];
          __syncwarp();
          ptx::tmem_ld_32x32b_x32(tmem + lane_off + (uint32_t)(half * BH + c_half + cc * 32), v);
          ptx::tmem_ld_wait();
          if (cc + 1 == BH / 64) {
            // this half's accumulator is in registers: the MMA may reuse it
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (rank == 0) ptx::mbar_arrive(&tempty[half]);
              else ptx::mbar_arrive_remote(tempty0 + (uint32_t)half * 8u);
            }
          }
          uint32_t pk[16];
          if (half == 0) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float u0 = __uint_as_float(v[2 * e]) * r;
              const float u1 = __uint_as_float(v[2 * e + 1]) * r;
              pk[e] = pack_bf16x2(lrelu_sq(u0, p.slope), lrelu_sq(u1, p.slope));
              g[cc * 16 + e] =
                  pack_bf16x2(lrelu_sq_grad(u0, p.slope) * r, lrelu_sq_grad(u1, p.slope) * r);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const uint32_t w = g[cc * 16 + e];
              pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * __uint_as_float(w << 16),
                                  __uint_as_float(v[2 * e + 1]) * __uint_as_float(w & 0xffff0000u));
            }
          }
          if (row0 < p.T)  // warp-uniform: boxes wholly past the last token are skipped
            store_box_bf16(half == 0 ? &tmA : &tmDu, wstg, stg_count, lane, pk, col0 + cc * 32,
                           row0);
        }
      }
      acc_phase ^= 1;
    }
    if (lane == 0) ptx::bulk_wait_group<0>();
    __syncwarp();
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (*s_abort && warp == 0 && lane == 0) {
    for (int s = 0; s < B_STAGES; ++s)
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
    ptx::tmem_dealloc_pair(tmem, 512);
  }
}

// dx = dy + dn' - r^2 x s, s = mean_i(dn'_i x_i), with dn' = (r du) W_gate^T.
// One warp per token row; lanes hold 16 of the 512 columns.
__global__ void __launch_bounds__(256) rmsnorm_bwd_kernel(const __nv_bfloat16* __restrict__ dnp,
                                                          const __nv_bfloat16* __restrict__ x,
                                                          const __nv_bfloat16* __restrict__ dy,
                                                          const float* __restrict__ rstd, int T,
                                                          __nv_bfloat16* __restrict__ dx) {
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const size_t base = (size_t)t * DM;
  float dn[16], xv[16];
  // lane owns columns [lane*8, lane*8+8) and [256 + lane*8, 256 + lane*8 + 8)
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c0 = h * 256 + lane * 8;
    const uint4 dq = __ldcs(reinterpret_cast<const uint4*>(dnp + base + c0));
    const __nv_bfloat162* dnh = reinterpret_cast<const __nv_bfloat162*>(&dq);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(dnh[e]);
      dn[h * 8 + 2 * e] = f.x;
      dn[h * 8 + 2 * e + 1] = f.y;
    }
    const uint4 xq = __ldg(reinterpret_cast<const uint4*>(x + base + c0));
    const __nv_bfloat162* xh = reinterpret_cast<const __nv_bfloat162*>(&xq);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(xh[e]);
      xv[h * 8 + 2 * e] = f.x;
      xv[h * 8 + 2 * e + 1] = f.y;
    }
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) s += dn[i] * xv[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  s /= (float)DM;
  const float r = rstd[t];
  const float k = r * r * s;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c0 = h * 256 + lane * 8;
    const uint4 dq = __ldg(reinterpret_cast<const uint4*>(dy + base + c0));
    const __nv_bfloat162* dh = reinterpret_cast<const __nv_bfloat162*>(&dq);
    uint4 o;
    uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(dh[e]);
      const int i0 = h * 8 + 2 * e;
      op[e] = pack_bf16x2(f.x + dn[i0] - k * xv[i0], f.y + dn[i0 + 1] - k * xv[i0 + 1]);
    }
    *reinterpret_cast<uint4*>(dx + base + c0) = o;
  }
}

}  // namespace

// ------------------------------------------------------------------ launchers

mlp_status launch_block_fwd(const void* x, const void* wg, const void* wd, int T, int hidden,
                            float eps, float slope, void* y, float* rstd, cudaStream_t st) {
  static bool configured = false;
  static int max_clusters = 0;
  if (!configured) {
    if (cudaFuncSetAttribute(block_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             F2_SMEM) != cudaSuccess)
      return MLP_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    cfg.blockDim = dim3(F2_THREADS);
    cfg.dynamicSmemBytes = F2_SMEM;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, block_fwd_kernel, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    max_clusters = n;
    configured = true;
  }
  CUtensorMap tx, tg, td;
  if (!encode_tmap_bf16_2d(&tx, x, DM, T, DM * 2, 64, F2_TOK)) return MLP_ERR_CUDA;
  if (!encode_tmap_bf16_2d(&tg, wg, hidden, DM, (unsigned long long)hidden * 2, 64, 128))
    return MLP_ERR_CUDA;
  if (!encode_tmap_bf16_2d(&td, wd, DM, hidden, DM * 2, 64, 64)) return MLP_ERR_CUDA;
  Fwd2Params p;
  p.T = T;
  p.n_chunks = hidden / F2_HC;
  p.tiles = (T + TM - 1) / TM;
  p.eps = eps;
  p.slope = slope;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.rstd = rstd;
  p.wait_ns = wait_limit_ns();
  p.err = device_error_word();
  if (!p.err) return MLP_ERR_CUDA;
  int clusters = max_clusters;
  if (clusters > p.tiles) clusters = p.tiles;
  if (clusters < 1) clusters = 1;
  LaunchScope ls("block_fwd", st, T, DM, hidden);
  launch_k(block_fwd_kernel, dim3(2 * clusters), dim3(F2_THREADS), F2_SMEM, st, tx, tg, td, p);
  return launch_status();
}

mlp_status launch_block_bwd_act(const void* x, const void* wg, const void* wd, const void* dy,
                                const float* rstd, int T, int hidden, float slope, void* a_out,
                                void* du_out, cudaStream_t st) {
  static bool configured = false;
  static int max_pairs = 0;
  if (!configured) {
    if (cudaFuncSetAttribute(block_bwd_act_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             B_SMEM) != cudaSuccess)
      return MLP_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    cfg.blockDim = dim3(B_THREADS);
    cfg.dynamicSmemBytes = B_SMEM;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, block_bwd_act_kernel, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    max_pairs = n;
    configured = true;
  }
  CUtensorMap tx, tg, tdy, twd, ta, tdu;
  if (!encode_tmap_bf16_2d(&tx, x, DM, T, DM * 2, 64, TM)) return MLP_ERR_CUDA;
  if (!encode_tmap_bf16_2d(&tg, wg, hidden, DM, (unsigned long long)hidden * 2, 64, 64))
    return MLP_ERR_CUDA;
  if (!encode_tmap_bf16_2d(&tdy, dy, DM, T, DM * 2, 64, TM)) return MLP_ERR_CUDA;
  if (!encode_tmap_bf16_2d(&twd, wd, DM, hidden, DM * 2, 64, BH / 2)) return MLP_ERR_CUDA;
  if (!encode_tmap_out_2d(&ta, a_out, 0, hidden, T, (unsigned long long)hidden * 2, 32, 32))
    return MLP_ERR_CUDA;
  if (!encode_tmap_out_2d(&tdu, du_out, 0, hidden, T, (unsigned long long)hidden * 2, 32, 32))
    return MLP_ERR_CUDA;
  BwdParams p;
  p.T = T;
  p.hidden = hidden;
  p.pairs_m = (T + 2 * TM - 1) / (2 * TM);
  p.tiles_h = hidden / BH;
  p.num_tiles = p.pairs_m * p.tiles_h;
  p.slope = slope;
  p.rstd = rstd;
  p.wait_ns = wait_limit_ns();
  p.err = device_error_word();
  if (!p.err) return MLP_ERR_CUDA;
  const int pairs = p.num_tiles < max_pairs ? p.num_tiles : max_pairs;
  LaunchScope ls("block_bwd_act", st, T, DM, hidden);
  launch_k(block_bwd_act_kernel, dim3(2 * pairs), dim3(B_THREADS), B_SMEM, st, tx, tg, tdy, twd, ta,
           tdu, p);
  return launch_status();
}

mlp_status launch_rmsnorm_bwd(const void* dnp, const void* x, const void* dy, const float* rstd,
                              int T, void* dx, cudaStream_t st) {
  if (T <= 0) return MLP_OK;
  LaunchScope ls("rmsnorm_bwd", st, T);
  launch_k(rmsnorm_bwd_kernel, dim3((T + 7) / 8), dim3(256), 0, st,
           static_cast<const __nv_bfloat16*>(dnp), static_cast<const __nv_bfloat16*>(x),
           static_cast<const __nv_bfloat16*>(dy), rstd, T, static_cast<__nv_bfloat16*>(dx));
  return launch_status();
}

}  // namespace mlp
