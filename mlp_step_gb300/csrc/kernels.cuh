// Host-side launchers of the library's kernels (one translation unit each),
// called by the C-ABI layer in api.cu.
#pragma once

#include <cuda.h>
#include "common.cuh"

namespace mlp {

// Segment map of the flat parameter buffer for the fused SGD + bf16 shadow
// refresh: segment k covers flat indices [flat_off[k], flat_off[k+1]) (the
// last one up to n); its elements form rows of `cols` values that land in the
// shadow at shadow_off[k] with a row pitch of cols_pad (shadow_off < 0: no
// shadow, e.g. biases).
struct SgdSegments {
  int n;
  long long flat_off[16];
  long long shadow_off[16];
  int cols[16];
  int cols_pad[16];
};

// k_elementwise.cu
// 16-bit buffers are bf16 or fp16: their format arguments (wb_fmt, dst_dtype,
// dl_dtype, dtype) take the MLP_DTYPE_* codes, MLP_DTYPE_F32 (0) meaning
// fp32 where a buffer may also be fp32.
mlp_status launch_sgd(float* w, const float* g, float* v, void* wb, int wb_fmt, long long n,
                      float lr, float mom, const SgdSegments& segs, cudaStream_t st);
mlp_status launch_shadow(const float* w, void* wb, int wb_fmt, long long n,
                         const SgdSegments& segs, cudaStream_t st);
mlp_status launch_cast_rows(const void* src, int src_dtype, void* dst, int dst_dtype, int rows,
                            int cols, int ld_dst, cudaStream_t st);
size_t xent_workspace_bytes(int B);
mlp_status launch_xent(const float* logits, int ldl, const int* labels, int B, int C,
                       float* loss_out, void* dlog, int dl_dtype, int ldd, int* argmax, void* ws,
                       cudaStream_t st);
size_t colsum_workspace_bytes(int rows, int cols);
mlp_status launch_colsum(const void* X, int dtype, int rows, int cols, int ld, float* out,
                         void* ws, cudaStream_t st);
size_t mse_ws_bytes(long long n);
mlp_status launch_mse(const void* y, const void* t, long long n, float* loss_out, void* dy,
                      void* ws, cudaStream_t st);
mlp_status launch_wait_selftest(unsigned long long limit_ns, cudaStream_t st);
// rstd[t] = 1 / sqrt(mean_i x[t][i]^2 + eps) for bf16 rows x [T][d] (d a
// multiple of 8, rows 16-byte aligned).
mlp_status launch_row_rstd(const void* x, long long T, int d, float eps, float* rstd,
                           cudaStream_t st);
// Sets column `col` of rows [0, rows) of each listed fp32 / bf16 / fp16 matrix to 1
// (and the columns after it, up to ld, to 0): the ones column that lets a
// weight-gradient GEMM produce the bias gradient as its last row.
struct OnesCols {
  int n;
  void* ptr[9];
  int ld[9];
  int col[9];
};
mlp_status launch_ones_cols(const OnesCols& oc, int rows, int dtype, cudaStream_t st);

// k_gemm_simt.cu: fp32 (or bf16-input) SIMT GEMM with the fused epilogue.
struct GemmArgs {
  int M, N, K;
  const void* A; int lda; int a_trans;
  const void* B; int ldb; int b_trans;
  const float* bias; int act;
  const void* mask; int ldm;
  void* C; int ldc; int c_bf16;  // c_bf16: C is 16-bit (bf16, or fp16 when f16 is set)
  // tensor-core path: A, B, the 16-bit outputs (C, xent_dlog, sgd_shadow) and
  // the ReLU mask are fp16 instead of bf16
  int f16 = 0;
  // optional scratch for split-K partial sums (tensor-core path only)
  void* ws = nullptr;
  size_t ws_bytes = 0;
  // Fused softmax cross entropy (tensor-core path; the whole problem must be
  // one tile: M <= 128, N <= 32): C receives the fp32 logits (nullable),
  // xent_dlog the bf16 dZ [M][xent_ldd], xent_loss the mean loss over
  // xent_norm rows, xent_argmax (nullable) the predictions.
  const int* xent_labels = nullptr;
  void* xent_dlog = nullptr;
  int xent_ldd = 0;
  float* xent_loss = nullptr;
  int* xent_argmax = nullptr;
  int xent_norm = 0;
  // Fused momentum SGD on the fp32 result g (tensor-core path): with w and v
  // laid out like C, v <- mom v - lr g, w <- w + v, and bf16(w) into
  // sgd_shadow[m][sgd_ld_shadow] for rows m < sgd_shadow_rows.  C still
  // receives g.
  float* sgd_w = nullptr;
  float* sgd_v = nullptr;
  float sgd_lr = 0.f, sgd_mom = 0.f;
  __nv_bfloat16* sgd_shadow = nullptr;
  int sgd_ld_shadow = 0;
  int sgd_shadow_rows = 0;
};
// fp32 operands (in_bf16 = 0) with g.ws holding gemm_simt_scratch_bytes()
// (16-byte aligned, its first 2 KiB zero before the first launch): small
// problems split K over more CTAs.
mlp_status launch_gemm_simt(const GemmArgs& g, int in_bf16, cudaStream_t st);
size_t gemm_simt_scratch_bytes();

// k_gemm_tc.cu: tcgen05 bf16 / fp16 GEMM (TMA-fed, fp32 accumulation in tensor
// memory).
mlp_status launch_gemm_tc(const GemmArgs& g, unsigned long long wait_ns, cudaStream_t st);
// k_gemm_tc.cu: the QKV projection of the fused attention preprocessing
// (g: bf16 x [M][K] times W_qkv [K][N], N = (n_q + 2 n_kv) * 64, bf16 C), with
// the per-token RMSNorm scale rstd, QK norm, partial RoPE over rope_dims (16,
// 32 or 64) and the q gain in the epilogue.
mlp_status launch_attn_prep_gemm(const GemmArgs& g, const float* rstd, const float* q_gain,
                                 int n_q, int n_kv, int rope_dims, int seq_len, float eps,
                                 float theta, cudaStream_t st);
// Scratch bytes a split-K launch of this shape would use (0: no split).
size_t gemm_tc_splitk_bytes(int M, int N, int K);

// k_gemm_tc.cu: one training step of a small MLP as ONE cooperative launch.
// Phase 0 optionally casts the input rows to bf16; then phases of mutually
// independent tensor-core GEMMs (bf16 operands, single-CTA 128 x 64 tiles,
// no split-K, fused epilogues as in launch_gemm_tc) run one after another,
// separated by grid-wide barriers, on one persistent CTA per SM.
constexpr int kStepMaxGemms = 24;
struct StepSpec {
  const void* cast_src = nullptr;
  int cast_dtype = 0;
  void* cast_dst = nullptr;  // 16-bit rows of pitch cast_ld (fp16 when f16 is set)
  int f16 = 0;
  // Optional second input buffer (same shape) for programs of several steps:
  // step s then reads buffer s % 2, and step s + 1's input is cast during
  // step s (by the CTAs idle in its smallest GEMM phase) instead of in a
  // phase of its own.  GEMMs whose A operand is cast_dst follow the buffer.
  void* cast_dst_alt = nullptr;
  int cast_rows = 0, cast_cols = 0, cast_ld = 0;
  int n_gemm = 0;
  GemmArgs gemm[kStepMaxGemms];
  int phase[kStepMaxGemms];  // >= 1, non-decreasing; equal phases run together
  // The program may run n_steps times back to back in the same launch (one
  // grid barrier between steps); step s reads the cast source at
  // cast_src + s * cast_stride bytes and its loss GEMM uses labels +
  // s * label_stride, loss + s * loss_stride, argmax + s * argmax_stride.
  int n_steps = 1;
  long long cast_stride = 0, label_stride = 0, loss_stride = 0, argmax_stride = 0;
};
// Whether launch_step_program can run this GEMM inside a step program.
bool step_gemm_supported(const GemmArgs& g);
// bar_words: one unsigned word of device memory owned by the caller (the
// grid barrier's arrival count, zeroed on the stream before each launch).
mlp_status launch_step_program(const StepSpec& s, unsigned* bar_words, unsigned long long wait_ns,
                               cudaStream_t st);

// k_block.cu: the MLP block (d = 512).
mlp_status launch_block_fwd(const void* x, const void* wg, const void* wd, int T, int hidden,
                            float eps, float slope, void* y, float* rstd, cudaStream_t st);
mlp_status launch_block_bwd_act(const void* x, const void* wg, const void* wd, const void* dy,
                                const float* rstd, int T, int hidden, float slope, void* a_out,
                                void* du_out, cudaStream_t st);
// dnp: bf16 [T][512]
mlp_status launch_rmsnorm_bwd(const void* dnp, const void* x, const void* dy, const float* rstd,
                              int T, void* dx, cudaStream_t st);

// Host helpers (api.cu)
unsigned long long wait_limit_ns();
// MLP_ORDER_LINEAR in effect (mlp_set_reduction_order)?
bool linear_order();
bool encode_tmap_bf16_2d(CUtensorMap* map, const void* base, unsigned long long inner,
                         unsigned long long outer, unsigned long long row_stride_bytes,
                         unsigned box_inner, unsigned box_outer);
// Same for an output tile map: bf16 (64-byte swizzle) or fp32 (128-byte
// swizzle) elements, box [box_outer][box_inner].
bool encode_tmap_out_2d(CUtensorMap* map, const void* base, int fp32, unsigned long long inner,
                        unsigned long long outer, unsigned long long row_stride_bytes,
                        unsigned box_inner, unsigned box_outer);

}  // namespace mlp
