// C-ABI entry points of the MLP block, the MSE loss and the block stack:
// argument checks, workspace carving and the enqueue order.
#include "kernels.cuh"
#include "trace.cuh"

using namespace mlp;

namespace {

inline cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool block_shape_ok(int T, int d, int hidden) {
  return T >= 0 && d == 512 && hidden >= 256 && hidden % 256 == 0 && hidden <= 65536;
}

struct BlockWs {
  size_t a, du, dn, split, total;
};

BlockWs block_ws(int T, int d, int hidden) {
  BlockWs w;
  w.a = align256((size_t)T * hidden * 2);
  w.du = align256((size_t)T * hidden * 2);
  w.dn = align256((size_t)T * d * 2);  // dn' in bf16
  // split-K partial sums of the two weight-gradient GEMMs (K = T)
  size_t s1 = gemm_tc_splitk_bytes(hidden, d, T), s2 = gemm_tc_splitk_bytes(d, hidden, T);
  w.split = align256(s1 > s2 ? s1 : s2);
  w.total = w.a + w.du + w.dn + w.split;
  return w;
}

mlp_status gemm(int M, int N, int K, const void* A, int lda, int a_trans, const void* B, int ldb,
                int b_trans, void* C, int ldc, cudaStream_t st, void* ws = nullptr,
                size_t ws_bytes = 0, int c_bf16 = 0) {
  GemmArgs g{};
  g.ws = ws;
  g.ws_bytes = ws_bytes;
  g.M = M; g.N = N; g.K = K;
  g.A = A; g.lda = lda; g.a_trans = a_trans;
  g.B = B; g.ldb = ldb; g.b_trans = b_trans;
  g.act = MLP_ACT_NONE;
  g.C = C; g.ldc = ldc; g.c_bf16 = c_bf16;
  return launch_gemm_tc(g, wait_limit_ns(), st);
}

// dx == nullptr: the weight gradients only (the input gradient of a stack's
// first block feeds nothing).
mlp_status block_bwd_impl(const void* x, const float* rstd, const void* wg, const void* wd,
                          const void* dy, int T, int d, int hidden, float slope, void* dx,
                          float* dwg, float* dwd, void* ws, cudaStream_t st) {
  const BlockWs w = block_ws(T, d, hidden);
  uint8_t* base = static_cast<uint8_t*>(ws);
  void* a_ws = base;
  void* du_ws = base + w.a;
  void* dn_ws = base + w.a + w.du;
  void* split_ws = base + w.a + w.du + w.dn;
  // a = f(u), r du, with u recomputed from x and rstd
  MLP_CHECK(launch_block_bwd_act(x, wg, wd, dy, rstd, T, hidden, slope, a_ws, du_ws, st));
  // dW_down = a^T dy   [hidden][d]
  MLP_CHECK(gemm(hidden, d, T, a_ws, hidden, 1, dy, d, 0, dwd, d, st, split_ws, w.split));
  // dW_gate = x^T (r du) = n^T du   [d][hidden]
  MLP_CHECK(gemm(d, hidden, T, x, d, 1, du_ws, hidden, 0, dwg, hidden, st, split_ws, w.split));
  if (!dx) return MLP_OK;
  // dn' = (r du) W_gate^T   [T][d], rounded to bf16 (it only feeds dx)
  MLP_CHECK(gemm(T, d, hidden, du_ws, hidden, 0, wg, hidden, 1, dn_ws, d, st, nullptr, 0, 1));
  // dx = dy + dn' - r^2 x mean(dn' x)
  return launch_rmsnorm_bwd(dn_ws, x, dy, rstd, T, dx, st);
}

}  // namespace

extern "C" {

size_t mlp_block_workspace_bytes(int T, int d, int hidden) {
  if (!block_shape_ok(T, d, hidden)) return 0;
  return block_ws(T, d, hidden).total;
}

mlp_status mlp_block_fwd(const void* x, const void* w_gate, const void* w_down, int T, int d,
                         int hidden, float eps, float slope, void* y, float* rstd_out,
                         void* stream) {
  NvtxRange nvtx_range("mlp_block_fwd");
  if (!block_shape_ok(T, d, hidden)) return T < 0 ? MLP_ERR_INVALID_ARG : MLP_ERR_UNSUPPORTED_SHAPE;
  if (!(eps >= 0.f)) return MLP_ERR_INVALID_ARG;
  if (T == 0) return MLP_OK;
  if (!x || !w_gate || !w_down || !y) return MLP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w_down) || !aligned16(y) ||
      (rstd_out && !aligned16(rstd_out)))
    return MLP_ERR_MISALIGNED;
  return launch_block_fwd(x, w_gate, w_down, T, hidden, eps, slope, y, rstd_out, S(stream));
}

mlp_status mlp_block_bwd(const void* x, const float* rstd, const void* w_gate,
                         const void* w_down, const void* dy, int T, int d, int hidden, float eps,
                         float slope, void* dx, float* dw_gate, float* dw_down, void* workspace,
                         size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("mlp_block_bwd");
  (void)eps;  // rstd carries the forward's normalisation
  if (!block_shape_ok(T, d, hidden)) return T < 0 ? MLP_ERR_INVALID_ARG : MLP_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MLP_OK;
  if (!x || !rstd || !w_gate || !w_down || !dy || !dx || !dw_gate || !dw_down || !workspace)
    return MLP_ERR_INVALID_ARG;
  if (ws_bytes < block_ws(T, d, hidden).total) return MLP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(rstd) || !aligned16(w_gate) || !aligned16(w_down) ||
      !aligned16(dy) || !aligned16(dx) || !aligned16(dw_gate) || !aligned16(dw_down) ||
      !aligned16(workspace))
    return MLP_ERR_MISALIGNED;
  return block_bwd_impl(x, rstd, w_gate, w_down, dy, T, d, hidden, slope, dx, dw_gate, dw_down,
                        workspace, S(stream));
}

size_t mlp_stack_param_count(int n_blocks, int d, int hidden) {
  if (n_blocks <= 0 || d <= 0 || hidden <= 0) return 0;
  return (size_t)n_blocks * 2 * d * hidden;
}

namespace {
struct StackWs {
  size_t xs, rstd, dy, dx, blk, mse, loss, total;
};
StackWs stack_ws(int n_blocks, int T, int d, int hidden) {
  StackWs w;
  w.xs = align256((size_t)n_blocks * T * d * 2);
  w.rstd = align256((size_t)n_blocks * T * 4);
  w.dy = align256((size_t)T * d * 2);
  w.dx = w.dy;
  w.blk = align256(block_ws(T, d, hidden).total);
  w.mse = align256(mse_ws_bytes((long long)T * d));
  w.loss = 256;
  w.total = w.xs + w.rstd + w.dy + w.dx + w.blk + w.mse + w.loss;
  return w;
}
}  // namespace

size_t mlp_stack_workspace_bytes(int n_blocks, int T, int d, int hidden) {
  if (n_blocks <= 0 || !block_shape_ok(T, d, hidden)) return 0;
  return stack_ws(n_blocks, T, d, hidden).total;
}

mlp_status mlp_stack_train_step(int n_blocks, int T, int d, int hidden, float eps, float slope,
                                const void* x0, const void* target, float* params,
                                float* velocity, float* grads, void* params_bf16, float lr,
                                float momentum, float* loss_out, void* workspace,
                                size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("mlp_stack_train_step");
  if (n_blocks <= 0 || T < 0) return MLP_ERR_INVALID_ARG;
  if (!block_shape_ok(T, d, hidden)) return MLP_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MLP_OK;
  if (!x0 || !target || !params || !velocity || !grads || !params_bf16 || !workspace)
    return MLP_ERR_INVALID_ARG;
  const StackWs w = stack_ws(n_blocks, T, d, hidden);
  if (ws_bytes < w.total) return MLP_ERR_INVALID_ARG;
  if (!aligned16(x0) || !aligned16(target) || !aligned16(params) || !aligned16(velocity) ||
      !aligned16(grads) || !aligned16(params_bf16) || !aligned16(workspace) ||
      (loss_out && !aligned16(loss_out)))
    return MLP_ERR_MISALIGNED;
  cudaStream_t st = S(stream);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(base);
  float* rstd = reinterpret_cast<float*>(base + w.xs);
  void* dy = base + w.xs + w.rstd;
  void* dx = base + w.xs + w.rstd + w.dy;
  void* blk = base + w.xs + w.rstd + w.dy + w.dx;
  void* mse = base + w.xs + w.rstd + w.dy + w.dx + w.blk;
  float* loss = loss_out ? loss_out
                         : reinterpret_cast<float*>(base + w.xs + w.rstd + w.dy + w.dx + w.blk +
                                                    w.mse);
  const size_t per = (size_t)2 * d * hidden;
  const size_t td = (size_t)T * d;
  const __nv_bfloat16* wb = static_cast<const __nv_bfloat16*>(params_bf16);
  // forward, saving every block input and rstd
  const void* cur = x0;
  for (int l = 0; l < n_blocks; ++l) {
    MLP_CHECK(launch_block_fwd(cur, wb + l * per, wb + l * per + (size_t)d * hidden, T, hidden,
                               eps, slope, xs + l * td, rstd + (size_t)l * T, st));
    cur = xs + l * td;
  }
  MLP_CHECK(launch_mse(cur, target, (long long)td, loss, dy, mse, st));
  for (int l = n_blocks - 1; l >= 0; --l) {
    const void* xin = l == 0 ? x0 : (const void*)(xs + (l - 1) * td);
    // the first block's input gradient is not an output of the step
    MLP_CHECK(block_bwd_impl(xin, rstd + (size_t)l * T, wb + l * per,
                             wb + l * per + (size_t)d * hidden, dy, T, d, hidden, slope,
                             l == 0 ? nullptr : dx, grads + l * per,
                             grads + l * per + (size_t)d * hidden, blk, st));
    void* t = dy;
    dy = dx;
    dx = t;
  }
  SgdSegments segs{};
  segs.n = 1;
  segs.flat_off[0] = 0;
  segs.shadow_off[0] = 0;
  segs.cols[0] = 1;
  segs.cols_pad[0] = 1;
  return launch_sgd(params, grads, velocity, params_bf16, MLP_DTYPE_BF16,
                    (long long)(per * n_blocks), lr, momentum, segs, st);
}

mlp_status mlp_attn_prep_fwd(const void* x, const void* w_qkv, const float* q_gain, int T,
                             int d, int n_q_heads, int n_kv_heads, int head_dim, int rope_dims,
                             int seq_len, float eps, float rope_theta, void* qkv_out,
                             float* rstd_out, void* stream) {
  NvtxRange nvtx_range("mlp_attn_prep_fwd");
  if (T < 0 || d <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || seq_len <= 0 || !(eps >= 0.f) ||
      !(rope_theta > 0.f))
    return MLP_ERR_INVALID_ARG;
  if (head_dim != 64 || (rope_dims != 16 && rope_dims != 32 && rope_dims != 64) || d % 8 != 0 ||
      d > 65536 || (long long)(n_q_heads + 2 * n_kv_heads) * 64 > 65536)
    return MLP_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MLP_OK;
  if (!x || !w_qkv || !q_gain || !qkv_out || !rstd_out) return MLP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_qkv) || !aligned16(qkv_out) || !aligned16(rstd_out) ||
      !aligned16(q_gain))
    return MLP_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MLP_CHECK(launch_row_rstd(x, T, d, eps, rstd_out, st));
  const int N = (n_q_heads + 2 * n_kv_heads) * 64;
  GemmArgs g{};
  g.M = T; g.N = N; g.K = d;
  g.A = x; g.lda = d; g.a_trans = 0;
  g.B = w_qkv; g.ldb = N; g.b_trans = 0;
  g.act = MLP_ACT_NONE;
  g.C = qkv_out; g.ldc = N; g.c_bf16 = 1;
  return launch_attn_prep_gemm(g, rstd_out, q_gain, n_q_heads, n_kv_heads, rope_dims, seq_len,
                               eps, rope_theta, st);
}

}  // extern "C"
