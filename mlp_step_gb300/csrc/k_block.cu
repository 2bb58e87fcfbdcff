// Transformer MLP block kernels for sm_103a ("Full-Depth MLP Megakernel +
// Fused Attention Preprocessing", "What Worked": RMSNorm -> gate projection ->
// LeakyReLU^2 -> down projection -> residual, the wide intermediate never
// written to memory).
//
// Forward (block_fwd_kernel): one CTA pair (a 2-CTA cluster) per 128-token
// tile.  Tensor memory of a CTA holds its half of the 128 x 512 fp32 output
// (256 columns) and two 128-column gate-chunk accumulators.  The 12 hidden
// chunks of 128 are split between the pair (CTA r computes chunks c with
// c % 2 == r): the gate MMA U_c = x W_gate[:, c] runs in tensor memory, the
// epilogue warps apply RMSNorm's row scale and LeakyReLU^2 in fp32, round to
// bf16 and write the activation chunk A_c into the operand slot of BOTH CTAs'
// shared memory (the peer's through distributed shared memory); both CTAs
// then accumulate y_half += A_c W_down[c, half].  So no FLOP is recomputed and
// the intermediate stays on chip (the page's design kept it in registers and
// lost to one large library GEMM; here it lives in tensor memory and shared
// memory and is fed to the tensor cores directly).
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

constexpr int TM = 128;                 // tokens per tile
constexpr int DM = 512;                 // model width
constexpr int HC = 128;                 // hidden chunk
constexpr int YH = 256;                 // output columns per CTA of the pair
constexpr int F_STAGES = 3;
constexpr int F_SLOTS = 2;                // one activation slot per CTA of the pair
constexpr int F_STAGE_BYTES = 49152;      // x k-block + two W_gate chunks' k-blocks
constexpr int F_SLOT_BYTES = TM * HC * 2;  // 32 KiB bf16 activation chunk
constexpr int F_SMEM = 1024 + F_SLOTS * F_SLOT_BYTES + F_STAGES * F_STAGE_BYTES + 2 * TM * 4 + 512;

__device__ __forceinline__ float lrelu_sq(float u, float slope) {
  const float t = u > 0.f ? u : slope * u;
  return t * t;
}

__device__ __forceinline__ float lrelu_sq_grad(float u, float slope) {
  return u > 0.f ? 2.f * u : 2.f * slope * slope * u;
}

struct FwdParams {
  int T, hidden, tiles, n_own;
  float eps, slope;
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  float* rstd;
  unsigned long long wait_ns;
  int* err;
};

constexpr int F_THREADS = 320;  // 10 warps

// MMA issue order of one tile for a CTA that owns n_own gate chunks (its
// chunks c = 2 j + rank, j = 0 .. n_own-1).  Gate chunks go in pairs: one
// N = 256 pass computes chunks j = 2p and 2p+1 into the two adjacent gate
// accumulators (operand reads per FLOP halve against two N = 128 passes),
// followed by the four down chunks c = 4p .. 4p+3 that those pairs of both
// CTAs feed.  An odd last chunk runs alone (N = 128).
enum : int { OP_GATE_PAIR = 0, OP_GATE = 1, OP_DOWN = 2 };
struct FwdOp {
  int kind, idx;
};
__device__ __forceinline__ int fwd_n_ops(int n_own) { return 5 * (n_own / 2) + 3 * (n_own & 1); }
__device__ __forceinline__ FwdOp fwd_op(int i, int n_own) {
  const int n_gp = n_own / 2;
  if (i < 5 * n_gp) {
    const int pr = i / 5, r = i % 5;
    if (r == 0) return {OP_GATE_PAIR, pr};
    return {OP_DOWN, 4 * pr + r - 1};
  }
  const int r = i - 5 * n_gp;
  if (r == 0) return {OP_GATE, n_own - 1};
  return {OP_DOWN, 2 * (n_own - 1) + r - 1};
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

// RMSNorm scale of the 32 token rows [row0, row0 + 32) of a tile, computed by
// one warp with coalesced loads (each row: lanes read 2 x 16 B); lane i
// returns the scale of row row0 + i (0 for rows past T).
__device__ __forceinline__ float warp_rows_rstd(const __nv_bfloat16* x, int row0, int T, float eps,
                                                int lane) {
  float mine = 0.f;
#pragma unroll 1
  for (int rr = 0; rr < 32; rr += 8) {
    uint4 v[8][2];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int m = row0 + rr + q;
      if (m < T) {
        const uint4* p = reinterpret_cast<const uint4*>(x + (size_t)m * DM);
        v[q][0] = __ldg(p + lane);
        v[q][1] = __ldg(p + 32 + lane);
      } else {
        v[q][0] = make_uint4(0, 0, 0, 0);
        v[q][1] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float ss = sumsq_bf16x8(v[q][0]) + sumsq_bf16x8(v[q][1]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == rr + q) mine = ss;
    }
  }
  return row0 + lane < T ? 1.0f / sqrtf(mine / (float)DM + eps) : 0.f;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(F_THREADS, 1)
    block_fwd_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmWg,
                     const __grid_constant__ CUtensorMap tmWd, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  // activation slots: chunk c lives in slot c % 2, the slot of its owner
  uint8_t* slots = smem;                                   // F_SLOTS x 32 KiB
  uint8_t* stages = smem + F_SLOTS * F_SLOT_BYTES;         // F_STAGES x 48 KiB
  float* rbuf = reinterpret_cast<float*>(stages + F_STAGES * F_STAGE_BYTES);  // [2][TM]
  uint64_t* full = reinterpret_cast<uint64_t*>(rbuf + 2 * TM);
  uint64_t* empty = full + F_STAGES;
  uint64_t* ufull = empty + F_STAGES;    // [2] gate accumulator ready
  uint64_t* uempty = ufull + 2;          // [2] gate accumulator drained (128 arrivals)
  uint64_t* afull = uempty + 2;          // [2] activation slot filled (1 arrival + copy bytes)
  uint64_t* aempty = afull + F_SLOTS;    // [2] slot consumed by both CTAs (2 arrivals)
  uint64_t* rready = aempty + F_SLOTS;   // [2] row scales of a tile in rbuf (128 arrivals)
  uint64_t* yfull = rready + 2;
  uint64_t* yempty = yfull + 1;          // 128 arrivals
  uint64_t* done = yempty + 1;
  uint64_t* awritten = done + 1;         // chunk stored in this CTA's slot (128 arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(awritten + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int cluster = blockIdx.x >> 1;
  const int n_clusters = gridDim.x >> 1;
  const int n_ops = fwd_n_ops(p.n_own);

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < F_STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&ufull[b], 1);
      ptx::mbar_init(&uempty[b], 128);
      ptx::mbar_init(&rready[b], 128);
    }
    for (int s2 = 0; s2 < F_SLOTS; ++s2) {
      ptx::mbar_init(&afull[s2], 1);
      ptx::mbar_init(&aempty[s2], 2);
    }
    ptx::mbar_init(yfull, 1);
    ptx::mbar_init(yempty, 128);
    ptx::mbar_init(done, 1);
    ptx::mbar_init(awritten, 128);
    *s_abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tmX);
    ptx::prefetch_tensormap(&tmWg);
    ptx::prefetch_tensormap(&tmWd);
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the peer's barriers are initialised before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // y half: cols [0,256); U buffers: [256,384), [384,512)
  pdl_wait();
  pdl_launch_dependents();

  int last_parity[F_STAGES];

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      for (int s = 0; s < F_STAGES; ++s) last_parity[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = cluster; t < p.tiles && ok && !*s_abort; t += n_clusters) {
        for (int i = 0; i < n_ops && ok; ++i) {
          const FwdOp op = fwd_op(i, p.n_own);
          const int nkb = op.kind == OP_DOWN ? HC / 64 : DM / 64;
          const uint32_t bytes = op.kind == OP_GATE_PAIR ? 49152u : 32768u;
          for (int kb = 0; kb < nkb; ++kb) {
            if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1, p.wait_ns, p.err,
                                        DEVERR_TIMEOUT_PRODUCER)) {
              *s_abort = 1;
              ok = false;
              break;
            }
            ptx::mbar_arrive_expect_tx(&full[stage], bytes);
            last_parity[stage] = (int)phase;
            uint8_t* st = stages + stage * F_STAGE_BYTES;
            if (op.kind == OP_DOWN) {
              const int c = op.idx;
#pragma unroll
              for (int j = 0; j < YH / 64; ++j)
                ptx::tma_load_2d(st + j * 8192, &tmWd, &full[stage], (int)rank * YH + j * 64,
                                 c * HC + kb * 64);
            } else {
              ptx::tma_load_2d(st, &tmX, &full[stage], kb * 64, t * TM);
              // chunk(s) c = 2 j + rank: one for a single gate, j = 2p, 2p+1 for a pair
              const int j0 = op.kind == OP_GATE_PAIR ? 2 * op.idx : op.idx;
              const int nch = op.kind == OP_GATE_PAIR ? 2 : 1;
              for (int q = 0; q < nch; ++q) {
                const int c = 2 * (j0 + q) + (int)rank;
                ptx::tma_load_2d(st + 16384 + q * 16384, &tmWg, &full[stage], c * HC, kb * 64);
                ptx::tma_load_2d(st + 24576 + q * 16384, &tmWg, &full[stage], c * HC + 64,
                                 kb * 64);
              }
            }
            if (++stage == F_STAGES) { stage = 0; phase ^= 1; }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc_g = ptx::idesc_bf16_f32(TM, HC, 0, 1);
      const uint32_t idesc_gp = ptx::idesc_bf16_f32(TM, 2 * HC, 0, 1);
      const uint32_t idesc_d = ptx::idesc_bf16_f32(TM, YH, 0, 1);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t ucount[2] = {0, 0}, acount[F_SLOTS] = {0, 0}, ycount = 0;
      bool ok = true;
      for (int t = cluster; t < p.tiles && ok && !*s_abort; t += n_clusters) {
        for (int i = 0; i < n_ops && ok; ++i) {
          const FwdOp op = fwd_op(i, p.n_own);
          if (op.kind != OP_DOWN) {
            // gate accumulators: a pair fills both, a single gate fills j % 2
            const bool pair = op.kind == OP_GATE_PAIR;
            const int b0 = pair ? 0 : (op.idx & 1);
            const int nb = pair ? 2 : 1;
            for (int q = 0; q < nb && ok; ++q) {
              const int b = b0 + q;
              if (!ptx::mbar_wait_bounded(&uempty[b], (ucount[b] & 1) ^ 1, p.wait_ns, p.err,
                                          DEVERR_TIMEOUT_MMA)) { ok = false; break; }
              ++ucount[b];
            }
            if (!ok) break;
            ptx::tc_fence_after();
            const uint32_t d = tmem + 256 + b0 * HC;
            const uint32_t idesc = pair ? idesc_gp : idesc_g;
            for (int kb = 0; kb < DM / 64; ++kb) {
              if (!ptx::mbar_wait_bounded(&full[stage], phase, p.wait_ns, p.err,
                                          DEVERR_TIMEOUT_MMA)) { ok = false; break; }
              ptx::tc_fence_after();
              const uint32_t sa = ptx::smem_u32(stages + stage * F_STAGE_BYTES);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t ad = ptx::sw128_desc(sa + k * 32, 16, 1024);
                const uint64_t bd = ptx::sw128_desc(sa + 16384 + k * 2048, 8192, 1024);
                ptx::mma_bf16(d, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
              }
              ptx::mma_commit(&empty[stage]);
              if (++stage == F_STAGES) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            for (int q = 0; q < nb; ++q) ptx::mma_commit(&ufull[b0 + q]);
          } else {
            const int c = op.idx;
            const int s = c & 1;
            if (c == 0) {
              if (!ptx::mbar_wait_bounded(yempty, (ycount & 1) ^ 1, p.wait_ns, p.err,
                                          DEVERR_TIMEOUT_MMA)) { ok = false; break; }
              ++ycount;
            }
            if (!ptx::mbar_wait_cluster_bounded(&afull[s], acount[s] & 1, p.wait_ns, p.err,
                                                DEVERR_TIMEOUT_PEER)) { ok = false; break; }
            ++acount[s];
            ptx::tc_fence_after();
            const uint32_t a_base = ptx::smem_u32(slots + s * F_SLOT_BYTES);
            for (int kb = 0; kb < HC / 64; ++kb) {
              if (!ptx::mbar_wait_bounded(&full[stage], phase, p.wait_ns, p.err,
                                          DEVERR_TIMEOUT_MMA)) { ok = false; break; }
              ptx::tc_fence_after();
              const uint32_t sb = ptx::smem_u32(stages + stage * F_STAGE_BYTES);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t ad = ptx::sw128_desc(a_base + kb * 16384 + k * 32, 16, 1024);
                const uint64_t bd = ptx::sw128_desc(sb + k * 2048, 8192, 1024);
                ptx::mma_bf16(tmem, ad, bd, idesc_d, (c > 0 || kb > 0 || k > 0) ? 1u : 0u);
              }
              ptx::mma_commit(&empty[stage]);
              if (++stage == F_STAGES) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            // slot s is reusable once both CTAs' MMAs that read it are done;
            // its owner (CTA s) waits for that
            ptx::mma_commit_multicast(&aempty[s], (uint16_t)(1u << s));
            if (c == 2 * p.n_own - 1) ptx::mma_commit(yfull);
          }
        }
      }
      if (!ok) *s_abort = 1;
      ptx::mma_commit(done);
      ptx::mbar_wait_bounded(done, 0, p.wait_ns, p.err, DEVERR_TIMEOUT_TEARDOWN);
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------------- activation warps
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint32_t uc[2] = {0, 0}, ac = 0, wc = 0;
    bool ok = true;
    int it = 0;
    for (int t = cluster; t < p.tiles && ok; t += n_clusters, ++it) {
      if (*s_abort) break;
      if (!ptx::mbar_wait_bounded(&rready[it & 1], (it >> 1) & 1, p.wait_ns, p.err,
                                  DEVERR_TIMEOUT_EPILOGUE)) { ok = false; break; }
      const float r = rbuf[(it & 1) * TM + row];
      for (int j = 0; j < p.n_own && ok; ++j) {
        const int b = j & 1;
        if (!ptx::mbar_wait_bounded(&ufull[b], uc[b] & 1, p.wait_ns, p.err,
                                    DEVERR_TIMEOUT_EPILOGUE)) { ok = false; break; }
        ++uc[b];
        // own chunk c = 2 j + rank goes to this CTA's slot
        const int sl = (int)rank;
        if (!ptx::mbar_wait_bounded(&aempty[sl], (ac & 1) ^ 1, p.wait_ns, p.err,
                                    DEVERR_TIMEOUT_EPILOGUE)) { ok = false; break; }
        ++ac;
        const uint32_t my_slot_addr = ptx::smem_u32(slots + sl * F_SLOT_BYTES);
        ptx::tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < HC / 32; ++cc) {
          uint32_t v[32];
          __syncwarp();
          ptx::tmem_ld_32x32b_x32(tmem + lane_off + 256 + b * HC + cc * 32, v);
          ptx::tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float a0 = lrelu_sq(__uint_as_float(v[2 * e]) * r, p.slope);
            const float a1 = lrelu_sq(__uint_as_float(v[2 * e + 1]) * r, p.slope);
            pk[e] = pack_bf16x2(a0, a1);
          }
          // K-major 128B-swizzled operand layout: 64-wide k blocks of
          // [128 rows][128 B]; 16-byte chunk j of row `row` sits at
          // chunk (j ^ (row & 7)).
          const int kb = cc >> 1;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int j16 = (cc & 1) * 4 + q;
            const uint32_t off =
                (uint32_t)(kb * 16384 + row * 128 + ((j16 ^ (row & 7)) << 4));
            ptx::st_shared_v4(my_slot_addr + off,
                              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]));
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&uempty[b]);
        // the chunk is complete in this CTA once all 128 writers are past
        // this point; one thread then publishes it locally and sends a copy
        // to the peer's slot (the copy's bytes complete the peer's barrier)
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(awritten);
        if (warp == 2 && lane == 0) {
          // on a timeout the chunk is not published; the peer and the MMA
          // warp then give up on their own bounded waits
          if (!ptx::mbar_wait_bounded(awritten, wc & 1, p.wait_ns, p.err,
                                      DEVERR_TIMEOUT_EPILOGUE)) {
            *s_abort = 1;
          } else {
          ptx::mbar_arrive(&afull[sl]);
          const uint32_t peer_bar = ptx::mapa_shared(ptx::smem_u32(&afull[sl]), peer);
          ptx::mbar_arrive_expect_tx_remote(peer_bar, (uint32_t)F_SLOT_BYTES);
          ptx::bulk_copy_to_peer(ptx::mapa_shared(my_slot_addr, peer), my_slot_addr,
                                 (uint32_t)F_SLOT_BYTES, peer_bar);
          }
        }
        ++wc;
      }
    }
    if (!ok) *s_abort = 1;
  } else {
    // ---------------------------------------------------------------- output warps
    // Row scales for the next tile are computed one tile ahead.  The residual
    // half-row of x streams through a ring of four 32-column chunks in
    // registers, the first four in flight while the tile's MMAs run.  (Ten
    // warps put three on some SM sub-partitions, which caps a thread at 168
    // registers, so the whole half-row cannot be held at once.)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint4 xq[4][4];
    uint32_t yc = 0;
    bool ok = true;
    int it = 0;
    auto publish_rstd = [&](int tile, int buf) {
      const float r = warp_rows_rstd(p.x, tile * TM + quarter * 32, p.T, p.eps, lane);
      rbuf[buf * TM + row] = r;
      const int m = tile * TM + row;
      if (rank == 0 && p.rstd && m < p.T) p.rstd[m] = r;
      ptx::mbar_arrive(&rready[buf]);
    };
    if (cluster < p.tiles) publish_rstd(cluster, 0);
    for (int t = cluster; t < p.tiles && ok; t += n_clusters, ++it) {
      if (*s_abort) break;
      const int tn = t + n_clusters;
      if (tn < p.tiles) publish_rstd(tn, (it + 1) & 1);
      const int m = t * TM + row;
      const bool valid = m < p.T;
      const uint4* xsrc = reinterpret_cast<const uint4*>(p.x + (size_t)m * DM + rank * YH);
      if (valid) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int q = 0; q < 4; ++q) xq[c][q] = __ldg(xsrc + c * 4 + q);
      }
      if (!ptx::mbar_wait_bounded(yfull, yc & 1, p.wait_ns, p.err, DEVERR_TIMEOUT_EPILOGUE)) {
        ok = false;
        break;
      }
      ++yc;
      ptx::tc_fence_after();
      uint4* yr = reinterpret_cast<uint4*>(p.y + (size_t)m * DM + rank * YH);
#pragma unroll
      for (int cc = 0; cc < YH / 32; ++cc) {
        uint32_t v[32];
        __syncwarp();
        ptx::tmem_ld_32x32b_x32(tmem + lane_off + cc * 32, v);
        ptx::tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const __nv_bfloat162* xh = reinterpret_cast<const __nv_bfloat162*>(&xq[cc & 3][q]);
            uint4 o;
            uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 xf = __bfloat1622float2(xh[e]);
              op[e] = pack_bf16x2(__uint_as_float(v[q * 8 + 2 * e]) + xf.x,
                                  __uint_as_float(v[q * 8 + 2 * e + 1]) + xf.y);
            }
            yr[cc * 4 + q] = o;
          }
          if (cc + 4 < YH / 32) {
#pragma unroll
            for (int q = 0; q < 4; ++q) xq[cc & 3][q] = __ldg(xsrc + (cc + 4) * 4 + q);
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(yempty);
    }
    if (!ok) *s_abort = 1;
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (*s_abort && warp == 0 && lane == 0) {
    for (int s = 0; s < F_STAGES; ++s)
      if (last_parity[s] >= 0)
        ptx::mbar_wait_bounded(&full[s], (uint32_t)last_parity[s], p.wait_ns, p.err,
                               DEVERR_TIMEOUT_TEARDOWN);
  }
  __syncwarp();
  __syncthreads();
  __syncwarp();
  // neither CTA leaves while the peer may still write into its shared memory
  ptx::cluster_sync();
  if (warp == 1) {
    __syncwarp();
    ptx::tmem_dealloc(tmem, 512);
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
  if (!configured) {
    if (cudaFuncSetAttribute(block_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             F_SMEM) != cudaSuccess)
      return MLP_ERR_CUDA;
    configured = true;
  }
  CUtensorMap tx, tg, td;
  if (!encode_tmap_bf16_2d(&tx, x, DM, T, DM * 2, 64, TM)) return MLP_ERR_CUDA;
  if (!encode_tmap_bf16_2d(&tg, wg, hidden, DM, (unsigned long long)hidden * 2, 64, 64))
    return MLP_ERR_CUDA;
  if (!encode_tmap_bf16_2d(&td, wd, DM, hidden, DM * 2, 64, 64)) return MLP_ERR_CUDA;
  FwdParams p;
  p.T = T;
  p.hidden = hidden;
  p.tiles = (T + TM - 1) / TM;
  p.n_own = hidden / (2 * HC);
  p.eps = eps;
  p.slope = slope;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.rstd = rstd;
  p.wait_ns = wait_limit_ns();
  p.err = device_error_word();
  if (!p.err) return MLP_ERR_CUDA;
  int clusters = num_sms() / 2;
  if (clusters > p.tiles) clusters = p.tiles;
  if (clusters < 1) clusters = 1;
  LaunchScope ls("block_fwd", st, T, DM, hidden);
  launch_k(block_fwd_kernel, dim3(2 * clusters), dim3(F_THREADS), F_SMEM, st, tx, tg, td, p);
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
