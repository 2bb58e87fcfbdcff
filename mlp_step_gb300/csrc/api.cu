// C-ABI entry points (include/mlp_step.h): argument checks, workspace
// carving, tensor-map encoding and the enqueue order of each step.  No
// arithmetic of the method lives here; every computation is a kernel launch.
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <utility>
#include <vector>
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "trace.cuh"

using namespace mlp;

namespace mlp {

// ------------------------------------------------------------ device error word

static __device__ int g_device_error = 0;

// Device address of the error word for the current device (looked up once per
// device; host code cannot use the symbol itself as a device pointer).
int* device_error_word() {
  static int* addr[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int*>(p);
  }
  return addr[dev];
}

// ------------------------------------------------------------ launch options

// Programmatic dependent launch is on unless MLP_STEP_PDL=0 is set in the
// environment (read once).
bool pdl_enabled() {
  static int on = -1;
  if (on < 0) {
    const char* e = getenv("MLP_STEP_PDL");
    on = (e && e[0] == '0') ? 0 : 1;
  }
  return on == 1;
}

// ------------------------------------------------------------ bounded waits

static unsigned long long g_wait_limit_ns = 0;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s

static int g_reduction_order = MLP_ORDER_FAST;
bool linear_order() { return g_reduction_order == MLP_ORDER_LINEAR; }

unsigned long long wait_limit_ns() {
  return g_wait_limit_ns ? g_wait_limit_ns : kDefaultWaitNs;
}

// ------------------------------------------------------------ tensor maps

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor [outer][inner] with the given row pitch; box
// [box_outer][box_inner] with 128-byte swizzle; out-of-range elements read 0.
bool encode_tmap_bf16_2d(CUtensorMap* map, const void* base, unsigned long long inner,
                         unsigned long long outer, unsigned long long row_stride_bytes,
                         unsigned box_inner, unsigned box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_out_2d(CUtensorMap* map, const void* base, int fp32, unsigned long long inner,
                        unsigned long long outer, unsigned long long row_stride_bytes,
                        unsigned box_inner, unsigned box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  fp32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace mlp

namespace {

inline cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline int round8(int x) { return (x + 7) / 8 * 8; }
inline int round64(int x) { return (x + 63) / 64 * 64; }
// Row pitch (elements) of bf16 matrices with n columns that TMA tiles read:
// compact for small heads, else whole 128-byte lines, so no box row of the
// tiles straddles two lines.
inline int bf16_pitch(int n) { return n <= 16 ? round8(n) : round64(n); }
// Row pitch of the handle's fp32 logits.
inline int f32_pitch(int n) { return n <= 16 ? n : (n + 31) / 32 * 32; }

// ------------------------------------------------------------ GEMM checks

mlp_status check_gemm(const GemmArgs& g, int in_dtype, int c_dtype) {
  if (g.M < 0 || g.N < 0 || g.K < 0) return MLP_ERR_INVALID_ARG;
  if (in_dtype != MLP_DTYPE_F32 && in_dtype != MLP_DTYPE_BF16 && in_dtype != MLP_DTYPE_F16)
    return MLP_ERR_INVALID_ARG;
  // 16-bit outputs take the operands' 16-bit type (bf16 for fp32 operands)
  const int c16 = in_dtype == MLP_DTYPE_F16 ? MLP_DTYPE_F16 : MLP_DTYPE_BF16;
  if (c_dtype != MLP_DTYPE_F32 && c_dtype != c16) return MLP_ERR_INVALID_ARG;
  if (g.act != MLP_ACT_NONE && g.act != MLP_ACT_RELU) return MLP_ERR_INVALID_ARG;
  if (g.M == 0 || g.N == 0) return MLP_OK;
  if (!g.C) return MLP_ERR_INVALID_ARG;
  if (g.K > 0 && (!g.A || !g.B)) return MLP_ERR_INVALID_ARG;
  // leading dimensions must cover the stored rows
  const int a_row = g.a_trans ? g.M : g.K;
  const int b_row = g.b_trans ? g.K : g.N;
  if (g.K > 0 && (g.lda < a_row || g.ldb < b_row)) return MLP_ERR_INVALID_ARG;
  if (g.ldc < g.N) return MLP_ERR_INVALID_ARG;
  if (g.mask && g.ldm < g.N) return MLP_ERR_INVALID_ARG;
  if (!aligned16(g.C) || (g.K > 0 && (!aligned16(g.A) || !aligned16(g.B))) ||
      (g.mask && !aligned16(g.mask)) || (g.bias && !aligned16(g.bias)))
    return MLP_ERR_MISALIGNED;
  if (in_dtype != MLP_DTYPE_F32 && g.K > 0) {
    // TMA: rows must start on 16-byte boundaries
    if (((long long)g.lda * 2) % 16 != 0 || ((long long)g.ldb * 2) % 16 != 0)
      return MLP_ERR_MISALIGNED;
    if ((long long)g.lda * 2 >= (1ll << 40) || (long long)g.ldb * 2 >= (1ll << 40))
      return MLP_ERR_UNSUPPORTED_SHAPE;
  }
  return MLP_OK;
}

mlp_status run_gemm(const GemmArgs& g, int in_bf16, cudaStream_t st) {
  if (in_bf16) return launch_gemm_tc(g, wait_limit_ns(), st);
  return launch_gemm_simt(g, 0, st);
}

// Launches the GEMM now, or (rec set) appends it to a step program in the
// given phase.
mlp_status issue_gemm(const GemmArgs& g, int in_bf16, cudaStream_t st, StepSpec* rec, int phase) {
  if (!rec) return run_gemm(g, in_bf16, st);
  if (rec->n_gemm >= kStepMaxGemms || !step_gemm_supported(g)) return MLP_ERR_UNSUPPORTED_SHAPE;
  rec->gemm[rec->n_gemm] = g;
  rec->phase[rec->n_gemm] = phase;
  ++rec->n_gemm;
  return MLP_OK;
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

const char* mlp_status_string(mlp_status s) {
  switch (s) {
    case MLP_OK: return "ok";
    case MLP_ERR_INVALID_ARG: return "invalid argument";
    case MLP_ERR_MISALIGNED: return "pointer or leading dimension not 16-byte aligned";
    case MLP_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MLP_ERR_CUDA: return "CUDA error";
    case MLP_ERR_DEVICE_TIMEOUT: return "a kernel abandoned a bounded wait";
    case MLP_ERR_NUMERIC: return "non-finite loss";
    default: return "unknown status";
  }
}

mlp_status mlp_get_device_status(void* stream) {
  if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return MLP_ERR_CUDA;
  int err = 0;
  if (cudaMemcpyFromSymbol(&err, g_device_error, sizeof(int)) != cudaSuccess) return MLP_ERR_CUDA;
  if (err != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return MLP_ERR_CUDA;
    return err == DEVERR_NUMERIC ? MLP_ERR_NUMERIC : MLP_ERR_DEVICE_TIMEOUT;
  }
  return MLP_OK;
}

void mlp_set_wait_limit_ns(long long ns) { g_wait_limit_ns = ns > 0 ? (unsigned long long)ns : 0; }

mlp_status mlp_set_reduction_order(int order) {
  if (order != MLP_ORDER_FAST && order != MLP_ORDER_LINEAR) return MLP_ERR_INVALID_ARG;
  g_reduction_order = order;
  return MLP_OK;
}

int mlp_get_reduction_order(void) { return g_reduction_order; }

mlp_status mlp_selftest_wait_timeout(long long limit_ns, void* stream) {
  if (limit_ns <= 0) return MLP_ERR_INVALID_ARG;
  return launch_wait_selftest((unsigned long long)limit_ns, S(stream));
}

// ------------------------------------------------------------ generic kernels

mlp_status mlp_gemm(int M, int N, int K, const void* A, int lda, int a_trans, const void* B,
                    int ldb, int b_trans, int in_dtype, const float* bias, int act,
                    const void* mask, int ldm, void* C, int ldc, int c_dtype, void* stream) {
  GemmArgs g{M, N, K, A, lda, a_trans ? 1 : 0, B, ldb, b_trans ? 1 : 0, bias, act, mask, ldm,
             C, ldc, c_dtype != MLP_DTYPE_F32 ? 1 : 0};
  g.f16 = in_dtype == MLP_DTYPE_F16 ? 1 : 0;
  MLP_CHECK(check_gemm(g, in_dtype, c_dtype));
  if (M == 0 || N == 0) return MLP_OK;
  return run_gemm(g, in_dtype != MLP_DTYPE_F32, S(stream));
}

size_t mlp_colsum_workspace_bytes(int rows, int cols) {
  if (rows <= 0 || cols <= 0) return 0;
  return colsum_workspace_bytes(rows, cols);
}

mlp_status mlp_colsum(const void* X, int dtype, int rows, int cols, int ld, float* out,
                      void* workspace, size_t ws_bytes, void* stream) {
  if (rows < 0 || cols < 0) return MLP_ERR_INVALID_ARG;
  if (dtype != MLP_DTYPE_F32 && dtype != MLP_DTYPE_BF16 && dtype != MLP_DTYPE_F16)
    return MLP_ERR_INVALID_ARG;
  if (cols == 0) return MLP_OK;
  if (!out || (rows > 0 && !X) || ld < cols) return MLP_ERR_INVALID_ARG;
  const size_t need = mlp_colsum_workspace_bytes(rows, cols);
  if (need > 0 && (!workspace || ws_bytes < need)) return MLP_ERR_INVALID_ARG;
  if ((X && !aligned16(X)) || !aligned16(out) || (workspace && !aligned16(workspace)))
    return MLP_ERR_MISALIGNED;
  return launch_colsum(X, dtype, rows, cols, ld, out, workspace, S(stream));
}

size_t softmax_xent_workspace_bytes(int batch, int classes) {
  (void)classes;
  return batch > 0 ? xent_workspace_bytes(batch) : 0;
}

mlp_status softmax_xent_fwd_bwd(const float* logits, int ld_logits, const int32_t* labels,
                                int batch, int classes, float* loss_out, void* dlogits,
                                int dlogits_dtype, int ld_dlogits, int32_t* argmax_out,
                                void* workspace, size_t ws_bytes, void* stream) {
  if (batch < 0 || classes <= 0) return MLP_ERR_INVALID_ARG;
  if (batch == 0) return MLP_OK;
  if (!logits || !labels || ld_logits < classes) return MLP_ERR_INVALID_ARG;
  if (dlogits && (ld_dlogits < classes ||
                  (dlogits_dtype != MLP_DTYPE_F32 && dlogits_dtype != MLP_DTYPE_BF16 &&
                   dlogits_dtype != MLP_DTYPE_F16)))
    return MLP_ERR_INVALID_ARG;
  const size_t need = softmax_xent_workspace_bytes(batch, classes);
  if (need > 0 && (!workspace || ws_bytes < need)) return MLP_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(labels) || (dlogits && !aligned16(dlogits)) ||
      (argmax_out && !aligned16(argmax_out)) || (loss_out && !aligned16(loss_out)) ||
      (workspace && !aligned16(workspace)))
    return MLP_ERR_MISALIGNED;
  return launch_xent(logits, ld_logits, labels, batch, classes, loss_out, dlogits,
                     dlogits ? dlogits_dtype : MLP_DTYPE_F32, ld_dlogits, argmax_out, workspace,
                     S(stream));
}

mlp_status sgd_momentum_step(float* w, const float* g, float* v, void* w_bf16, size_t n,
                             float lr, float momentum, void* stream) {
  if (n == 0) return MLP_OK;
  if (!w || !g || !v) return MLP_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(g) || !aligned16(v) || (w_bf16 && !aligned16(w_bf16)))
    return MLP_ERR_MISALIGNED;
  SgdSegments segs{};
  segs.n = 1;
  segs.flat_off[0] = 0;
  segs.shadow_off[0] = w_bf16 ? 0 : -1;
  segs.cols[0] = 1;
  segs.cols_pad[0] = 1;
  return launch_sgd(w, g, v, w_bf16, MLP_DTYPE_BF16, (long long)n, lr, momentum, segs,
                    S(stream));
}

size_t mse_workspace_bytes(size_t n) { return n ? mse_ws_bytes((long long)n) : 0; }

mlp_status mse_loss_fwd_bwd(const void* y, const void* t, size_t n, float* loss_out, void* dy,
                            void* workspace, size_t ws_bytes, void* stream) {
  if (n == 0) return MLP_OK;
  if (!y || !t || !workspace || ws_bytes < mse_workspace_bytes(n)) return MLP_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(t) || (dy && !aligned16(dy)) || !aligned16(workspace) ||
      (loss_out && !aligned16(loss_out)))
    return MLP_ERR_MISALIGNED;
  return launch_mse(y, t, (long long)n, loss_out, dy, workspace, S(stream));
}

}  // extern "C"

// ====================================================================== MLP handle

struct mlp_handle {
  std::vector<int> dims;
  int L = 0;
  int act = MLP_ACT_RELU;
  int prec = MLP_PREC_FP32;
  int max_batch = 0;
  float* params = nullptr;
  float* velocity = nullptr;
  float* grads = nullptr;
  __nv_bfloat16* shadow = nullptr;  // 16-bit weight shadow (bf16 bits, or fp16 for MLP_PREC_FP16)
  long long n_params = 0;
  std::vector<long long> w_off, b_off, shadow_off;
  std::vector<int> out_pad;        // shadow row pitch per layer
  // Layer inputs (X and every hidden activation) are stored with one extra
  // column of ones after the features (ld = width + 1 rounded up to 64
  // elements, so rows start on 128-byte lines for the TMA tiles): the
  // weight-gradient GEMM over [In | 1] then yields [dW; db], which is exactly
  // the flat layout of W followed by b.
  std::vector<int> act_ld;         // act_ld[l]: pitch of layer l's input buffer
  void* x_copy = nullptr;          // [max_batch][act_ld[0]]
  void* x_copy_alt = nullptr;      // second input buffer of multi-step programs (16-bit only)
  void* simt_ws = nullptr;         // split-K scratch of the fp32 GEMMs (fp32 only)
  std::vector<void*> acts;         // acts[l] = H_{l+1}, l = 0..L-2
  float* logits = nullptr;         // [max_batch][C]
  void* dlogits = nullptr;         // [max_batch][ldz]
  int ldz = 0;
  int ldl = 0;                     // row pitch of logits
  void* dh[2] = {nullptr, nullptr};
  float* loss = nullptr;
  unsigned* step_bar = nullptr;    // grid barrier words of the step program (in the loss block)
  void* red = nullptr;             // reduction partials
  size_t red_bytes = 0;
  SgdSegments segs{};
  bool ones_ready = false;
  bool have_forward = false;
};

namespace {

int esz(int prec) { return prec == MLP_PREC_FP32 ? 4 : 2; }

// The tensor-core path (bf16 or fp16 operands)?
bool tc_prec(int prec) { return prec == MLP_PREC_BF16 || prec == MLP_PREC_FP16; }

// MLP_DTYPE_* code of the handle's operand buffers (input copy, hidden
// activations, dZ / dH, weight shadow).
int buf_dtype(const mlp_handle* h) {
  return h->prec == MLP_PREC_FP16 ? MLP_DTYPE_F16
                                  : (h->prec == MLP_PREC_BF16 ? MLP_DTYPE_BF16 : MLP_DTYPE_F32);
}

bool dims_ok(const int* dims, int n_dims) {
  if (!dims || n_dims < 2 || n_dims > 9) return false;
  for (int i = 0; i < n_dims; ++i)
    if (dims[i] <= 0) return false;
  return true;
}

struct Plan {
  size_t x, x_alt, acts_total, logits, dlogits, dh, loss, red, simt, total;
};

Plan plan(const int* dims, int n_dims, int max_batch, int prec) {
  Plan p{};
  const int L = n_dims - 1;
  const size_t B = (size_t)max_batch;
  const int e = esz(prec);
  p.x = align256(B * round64(dims[0] + 1) * e);
  p.x_alt = tc_prec(prec) ? p.x : 0;
  p.acts_total = 0;
  int maxh = 8;
  for (int l = 1; l < L; ++l) {
    p.acts_total += align256(B * round64(dims[l] + 1) * e);
    if (round64(dims[l] + 1) > maxh) maxh = round64(dims[l] + 1);
  }
  if (round64(dims[0] + 1) > maxh) maxh = round64(dims[0] + 1);
  p.logits = align256(B * f32_pitch(dims[L]) * sizeof(float));
  p.dlogits = align256(B * bf16_pitch(dims[L]) * e);
  p.dh = align256(B * maxh * e);
  p.loss = 256;
  size_t red = xent_workspace_bytes(max_batch);
  p.red = align256(red > 0 ? red : 256);
  p.simt = tc_prec(prec) ? 0 : align256(gemm_simt_scratch_bytes());
  p.total = p.x + p.x_alt + p.acts_total + p.logits + p.dlogits + 2 * p.dh + p.loss + p.red +
            p.simt;
  return p;
}

// ones columns of every layer input buffer, for all max_batch rows (once per
// handle: the forward GEMMs never write them)
mlp_status ensure_ones(mlp_handle* h, cudaStream_t st) {
  if (h->ones_ready) return MLP_OK;
  OnesCols oc{};
  oc.n = h->L;
  oc.ptr[0] = h->x_copy;
  oc.ld[0] = h->act_ld[0];
  oc.col[0] = h->dims[0];
  for (int l = 1; l < h->L; ++l) {
    oc.ptr[l] = h->acts[l - 1];
    oc.ld[l] = h->act_ld[l];
    oc.col[l] = h->dims[l];
  }
  if (h->x_copy_alt) {
    oc.ptr[oc.n] = h->x_copy_alt;
    oc.ld[oc.n] = h->act_ld[0];
    oc.col[oc.n] = h->dims[0];
    ++oc.n;
  }
  MLP_CHECK(launch_ones_cols(oc, h->max_batch, buf_dtype(h), st));
  // the split-K counters of the fp32 GEMMs start at zero (each launch leaves
  // them so)
  if (h->simt_ws && cudaMemsetAsync(h->simt_ws, 0, 4096, st) != cudaSuccess) return MLP_ERR_CUDA;
  h->ones_ready = true;
  return MLP_OK;
}

// fp32 GEMMs of the handle get its split-K scratch
GemmArgs& with_simt_ws(const mlp_handle* h, GemmArgs& g) {
  if (!tc_prec(h->prec) && h->simt_ws) {
    g.ws = h->simt_ws;
    g.ws_bytes = gemm_simt_scratch_bytes();
  }
  return g;
}

// Hidden layers 0 .. L-2 of the forward (bias + activation in the epilogue);
// in a step program, layer l is phase 1 + l.
mlp_status forward_hidden(mlp_handle* h, int batch, cudaStream_t st, StepSpec* rec = nullptr) {
  const bool bf = tc_prec(h->prec);
  for (int l = 0; l + 1 < h->L; ++l) {
    GemmArgs g{};
    g.f16 = h->prec == MLP_PREC_FP16 ? 1 : 0;
    g.M = batch;
    g.N = h->dims[l + 1];
    g.K = h->dims[l];
    g.A = l == 0 ? h->x_copy : h->acts[l - 1];
    g.lda = h->act_ld[l];
    g.a_trans = 0;
    if (bf) {
      g.B = h->shadow + h->shadow_off[l];
      g.ldb = h->out_pad[l];
    } else {
      g.B = h->params + h->w_off[l];
      g.ldb = h->dims[l + 1];
    }
    g.b_trans = 0;
    g.bias = h->params + h->b_off[l];
    g.act = h->act;
    g.C = h->acts[l];
    g.ldc = h->act_ld[l + 1];
    g.c_bf16 = bf ? 1 : 0;
    MLP_CHECK(issue_gemm(with_simt_ws(h, g), bf, st, rec, 1 + l));
  }
  return MLP_OK;
}

// The output layer's GEMM operands (logits = In W_L + b_L).
GemmArgs logits_gemm(mlp_handle* h, int batch, float* logits, int ld_logits) {
  const bool bf = tc_prec(h->prec);
  const int l = h->L - 1;
  GemmArgs g{};
  g.f16 = h->prec == MLP_PREC_FP16 ? 1 : 0;
  g.M = batch;
  g.N = h->dims[l + 1];
  g.K = h->dims[l];
  g.A = l == 0 ? h->x_copy : h->acts[l - 1];
  g.lda = h->act_ld[l];
  if (bf) {
    g.B = h->shadow + h->shadow_off[l];
    g.ldb = h->out_pad[l];
  } else {
    g.B = h->params + h->w_off[l];
    g.ldb = h->dims[l + 1];
  }
  g.bias = h->params + h->b_off[l];
  g.act = MLP_ACT_NONE;
  g.C = logits;
  g.ldc = ld_logits;
  g.c_bf16 = 0;
  return g;
}

mlp_status load_input(mlp_handle* h, const void* x, int x_dtype, int batch, cudaStream_t st) {
  MLP_CHECK(ensure_ones(h, st));
  // X goes into the workspace copy with the ones column, in the path's type
  const int d0 = h->dims[0];
  // rows of d0 values into rows of pitch act_ld[0]
  return launch_cast_rows(x, x_dtype, h->x_copy, buf_dtype(h), batch, d0, h->act_ld[0], st);
}

// Backward from dY = dlogits.  With fuse_sgd, each layer's weight-gradient
// GEMM also applies momentum SGD to that layer's weights and bias (after the
// layer's input gradient has read the old weights).  In a step program
// (after the forward's phases 1 .. L), layer l's input gradient is phase
// 2L - l and its weight gradient the phase after (or, without an input
// gradient, the phase after its dY's): each reads only earlier phases'
// outputs and the weights it reads are updated in a later phase.
mlp_status backward_impl(mlp_handle* h, const void* dlogits, int ld_dlogits, int batch, void* dx,
                         bool fuse_sgd, float lr, float mom, cudaStream_t st,
                         StepSpec* rec = nullptr) {
  const bool bf = tc_prec(h->prec);
  const int f16 = h->prec == MLP_PREC_FP16 ? 1 : 0;
  const void* dY = dlogits;
  int ld_dy = ld_dlogits;
  for (int l = h->L - 1; l >= 0; --l) {
    const int fi = h->dims[l], fo = h->dims[l + 1];
    const void* in = l == 0 ? h->x_copy : h->acts[l - 1];
    const int ld_in = h->act_ld[l];
    // dIn = (dY W_l^T) * (H_l > 0)   (B = W_l read transposed); reads the
    // layer's weights before any update
    GemmArgs gd{};
    gd.f16 = f16;
    const bool want_din = l > 0 || dx;
    if (want_din) {
      gd.M = batch; gd.N = fi; gd.K = fo;
      gd.A = dY; gd.lda = ld_dy; gd.a_trans = 0;
      if (bf) { gd.B = h->shadow + h->shadow_off[l]; gd.ldb = h->out_pad[l]; }
      else { gd.B = h->params + h->w_off[l]; gd.ldb = fo; }
      gd.b_trans = 1;
      gd.act = MLP_ACT_NONE;
      if (l > 0) {
        gd.mask = h->act == MLP_ACT_RELU ? h->acts[l - 1] : nullptr;
        gd.ldm = h->act_ld[l];
        gd.C = h->dh[l & 1];
        gd.ldc = h->act_ld[l];
      } else {
        gd.C = dx;
        gd.ldc = fi;
      }
      gd.c_bf16 = bf ? 1 : 0;
      MLP_CHECK(issue_gemm(with_simt_ws(h, gd), bf, st, rec, 2 * h->L - l));
    }
    // [dW_l; db_l] = [In_l | 1]^T dY_l   (A = In_l read transposed), written
    // over the layer's flat slice of grads
    GemmArgs gw{};
    gw.f16 = f16;
    gw.M = fi + 1; gw.N = fo; gw.K = batch;
    gw.A = in; gw.lda = ld_in; gw.a_trans = 1;
    gw.B = dY; gw.ldb = ld_dy; gw.b_trans = 0;
    gw.C = h->grads + h->w_off[l]; gw.ldc = fo; gw.c_bf16 = 0;
    gw.act = MLP_ACT_NONE;
    // The update rides in the GEMM epilogue only for small weight matrices:
    // there it saves a launch; on large ones the epilogue's per-row accesses
    // to w and v compete with the MMA operand traffic and the flat SGD kernel
    // (which streams at HBM speed) is faster.
    const bool fuse_here = fuse_sgd && (long long)(fi + 1) * fo <= (1ll << 18);
    if (fuse_here) {
      gw.sgd_w = h->params + h->w_off[l];
      gw.sgd_v = h->velocity + h->w_off[l];
      gw.sgd_lr = lr;
      gw.sgd_mom = mom;
      gw.sgd_shadow = h->shadow ? h->shadow + h->shadow_off[l] : nullptr;
      gw.sgd_ld_shadow = h->out_pad[l];
      gw.sgd_shadow_rows = fi;
    }
    if (rec && fuse_sgd && !fuse_here) return MLP_ERR_UNSUPPORTED_SHAPE;
    MLP_CHECK(issue_gemm(with_simt_ws(h, gw), bf, st, rec, 2 * h->L - l + (want_din ? 1 : 0)));
    if (fuse_sgd && !fuse_here) {
      // flat SGD over this layer's W and b (and its shadow rows)
      SgdSegments seg{};
      seg.n = 2;
      seg.flat_off[0] = 0;
      seg.shadow_off[0] = h->shadow ? 0 : -1;
      seg.cols[0] = fo;
      seg.cols_pad[0] = h->out_pad[l];
      seg.flat_off[1] = (long long)fi * fo;
      seg.shadow_off[1] = -1;
      seg.cols[1] = 1;
      seg.cols_pad[1] = 1;
      MLP_CHECK(launch_sgd(h->params + h->w_off[l], h->grads + h->w_off[l],
                           h->velocity + h->w_off[l],
                           h->shadow ? h->shadow + h->shadow_off[l] : nullptr, buf_dtype(h),
                           (long long)(fi + 1) * fo, lr, mom, seg, st));
    }
    if (l > 0) {
      dY = gd.C;
      ld_dy = gd.ldc;
    }
  }
  return MLP_OK;
}

// The step program of one training step (bf16 path, one-tile head): input
// cast (phase 0), forward, logits with the softmax cross entropy, backward
// with momentum SGD in every weight-gradient GEMM -- the same kernels'
// arithmetic in the same order as the launch-per-GEMM path.  False when some
// GEMM does not fit one round of CTAs or a layer's update cannot ride in its
// gradient GEMM.
bool build_step_spec(mlp_handle* h, const void* x, int x_dtype, const int32_t* labels, int batch,
                     float lr, float momentum, float* loss, int32_t* argmax_out, cudaStream_t st,
                     StepSpec* spec) {
  const int C = h->dims[h->L];
  if (!tc_prec(h->prec) || batch > 128 || C > 32) return false;
  spec->f16 = h->prec == MLP_PREC_FP16 ? 1 : 0;
  spec->cast_src = x;
  spec->cast_dtype = x_dtype;
  spec->cast_dst = h->x_copy;
  spec->cast_rows = batch;
  spec->cast_cols = h->dims[0];
  spec->cast_ld = h->act_ld[0];
  if (forward_hidden(h, batch, st, spec) != MLP_OK) return false;
  GemmArgs gz = logits_gemm(h, batch, h->logits, h->ldl);
  gz.xent_labels = labels;
  gz.xent_dlog = h->dlogits;
  gz.xent_ldd = h->ldz;
  gz.xent_loss = loss;
  gz.xent_argmax = argmax_out;
  gz.xent_norm = batch;
  if (issue_gemm(gz, true, st, spec, h->L) != MLP_OK) return false;
  return backward_impl(h, h->dlogits, h->ldz, batch, nullptr, true, lr, momentum, st, spec) ==
         MLP_OK;
}

mlp_status train_step_impl(mlp_handle* h, const void* x, int x_dtype, const int32_t* labels,
                           int batch, float lr, float momentum, float* loss_out,
                           int32_t* argmax_out, cudaStream_t st) {
  const int C = h->dims[h->L];
  const bool bf = tc_prec(h->prec);
  float* loss = loss_out ? loss_out : h->loss;
  {
    // the whole step as one cooperative launch where it fits
    StepSpec spec;
    if (build_step_spec(h, x, x_dtype, labels, batch, lr, momentum, loss, argmax_out, st, &spec)) {
      MLP_CHECK(ensure_ones(h, st));
      MLP_CHECK(launch_step_program(spec, h->step_bar, wait_limit_ns(), st));
      h->have_forward = true;
      return MLP_OK;
    }
  }
  MLP_CHECK(load_input(h, x, x_dtype, batch, st));
  MLP_CHECK(forward_hidden(h, batch, st));
  GemmArgs gz = logits_gemm(h, batch, h->logits, h->ldl);
  if (bf && batch <= 128 && C <= 32) {
    // one tile holds the whole head: softmax cross entropy in its epilogue
    gz.xent_labels = labels;
    gz.xent_dlog = h->dlogits;
    gz.xent_ldd = h->ldz;
    gz.xent_loss = loss;
    gz.xent_argmax = argmax_out;
    gz.xent_norm = batch;
    MLP_CHECK(run_gemm(gz, true, st));
  } else {
    MLP_CHECK(run_gemm(with_simt_ws(h, gz), bf, st));
    MLP_CHECK(launch_xent(h->logits, h->ldl, labels, batch, C, loss, h->dlogits, buf_dtype(h),
                          h->ldz, argmax_out, h->red, st));
  }
  h->have_forward = true;
  if (bf) return backward_impl(h, h->dlogits, h->ldz, batch, nullptr, true, lr, momentum, st);
  MLP_CHECK(backward_impl(h, h->dlogits, h->ldz, batch, nullptr, false, 0.f, 0.f, st));
  return mlp_sgd_step(h, lr, momentum, st);
}

}  // namespace

extern "C" {

size_t mlp_param_count(const int* dims, int n_dims) {
  if (!dims_ok(dims, n_dims)) return 0;
  size_t n = 0;
  for (int l = 0; l + 1 < n_dims; ++l) n += (size_t)dims[l] * dims[l + 1] + dims[l + 1];
  return n;
}

size_t mlp_param_offset(const int* dims, int n_dims, int layer, int which) {
  if (!dims_ok(dims, n_dims) || layer < 0 || layer >= n_dims - 1 || (which != 0 && which != 1))
    return (size_t)-1;
  size_t off = 0;
  for (int l = 0; l < layer; ++l) off += (size_t)dims[l] * dims[l + 1] + dims[l + 1];
  if (which == 1) off += (size_t)dims[layer] * dims[layer + 1];
  return off;
}

size_t mlp_shadow_elems(const int* dims, int n_dims) {
  if (!dims_ok(dims, n_dims)) return 0;
  size_t n = 0;
  for (int l = 0; l + 1 < n_dims; ++l) n += (size_t)dims[l] * bf16_pitch(dims[l + 1]);
  return n;
}

size_t mlp_workspace_bytes(const int* dims, int n_dims, int max_batch, int prec) {
  if (!dims_ok(dims, n_dims) || max_batch <= 0) return 0;
  return plan(dims, n_dims, max_batch, prec).total;
}

mlp_status mlp_create(const int* dims, int n_dims, int hidden_act, int prec, int max_batch,
                      float* params, float* velocity, float* grads, void* params_bf16,
                      void* workspace, size_t ws_bytes, mlp_handle** out) {
  if (!out) return MLP_ERR_INVALID_ARG;
  *out = nullptr;
  if (!dims_ok(dims, n_dims) || max_batch <= 0) return MLP_ERR_INVALID_ARG;
  if (prec != MLP_PREC_FP32 && prec != MLP_PREC_BF16 && prec != MLP_PREC_FP16)
    return MLP_ERR_INVALID_ARG;
  if (hidden_act != MLP_ACT_RELU && hidden_act != MLP_ACT_NONE) return MLP_ERR_INVALID_ARG;
  if (!params || !velocity || !grads || !workspace) return MLP_ERR_INVALID_ARG;
  if (tc_prec(prec) && !params_bf16) return MLP_ERR_INVALID_ARG;
  const Plan pl = plan(dims, n_dims, max_batch, prec);
  if (ws_bytes < pl.total) return MLP_ERR_INVALID_ARG;
  if (!aligned16(params) || !aligned16(velocity) || !aligned16(grads) || !aligned16(workspace) ||
      (params_bf16 && !aligned16(params_bf16)))
    return MLP_ERR_MISALIGNED;

  mlp_handle* h = new (std::nothrow) mlp_handle();
  if (!h) return MLP_ERR_INVALID_ARG;
  h->dims.assign(dims, dims + n_dims);
  h->L = n_dims - 1;
  h->act = hidden_act;
  h->prec = prec;
  h->max_batch = max_batch;
  h->params = params;
  h->velocity = velocity;
  h->grads = grads;
  h->shadow = tc_prec(prec) ? static_cast<__nv_bfloat16*>(params_bf16) : nullptr;
  h->n_params = (long long)mlp_param_count(dims, n_dims);
  long long off = 0, soff = 0;
  for (int l = 0; l < h->L; ++l) {
    h->w_off.push_back(off);
    off += (long long)dims[l] * dims[l + 1];
    h->b_off.push_back(off);
    off += dims[l + 1];
    h->shadow_off.push_back(soff);
    h->out_pad.push_back(bf16_pitch(dims[l + 1]));
    soff += (long long)dims[l] * bf16_pitch(dims[l + 1]);
  }
  for (int l = 0; l < h->L; ++l) h->act_ld.push_back(round64(dims[l] + 1));
  // segment map for the fused SGD + shadow refresh
  h->segs.n = 2 * h->L;
  for (int l = 0; l < h->L; ++l) {
    h->segs.flat_off[2 * l] = h->w_off[l];
    h->segs.shadow_off[2 * l] = h->shadow ? h->shadow_off[l] : -1;
    h->segs.cols[2 * l] = dims[l + 1];
    h->segs.cols_pad[2 * l] = h->out_pad[l];
    h->segs.flat_off[2 * l + 1] = h->b_off[l];
    h->segs.shadow_off[2 * l + 1] = -1;
    h->segs.cols[2 * l + 1] = 1;
    h->segs.cols_pad[2 * l + 1] = 1;
  }
  // workspace carving
  uint8_t* w = static_cast<uint8_t*>(workspace);
  const int e = esz(prec);
  const size_t B = (size_t)max_batch;
  h->x_copy = w;
  w += pl.x;
  if (pl.x_alt) {
    h->x_copy_alt = w;
    w += pl.x_alt;
  }
  for (int l = 1; l < h->L; ++l) {
    h->acts.push_back(w);
    w += align256(B * h->act_ld[l] * e);
  }
  h->logits = reinterpret_cast<float*>(w);
  w += pl.logits;
  h->ldz = bf16_pitch(dims[h->L]);
  h->ldl = f32_pitch(dims[h->L]);
  h->dlogits = w;
  w += pl.dlogits;
  h->dh[0] = w;
  w += pl.dh;
  h->dh[1] = w;
  w += pl.dh;
  h->loss = reinterpret_cast<float*>(w);
  h->step_bar = reinterpret_cast<unsigned*>(w + 128);
  w += pl.loss;
  h->red = w;
  h->red_bytes = pl.red;
  w += pl.red;
  if (pl.simt) h->simt_ws = w;
  *out = h;
  return MLP_OK;
}

void mlp_destroy(mlp_handle* h) { delete h; }

mlp_status mlp_refresh_shadow(mlp_handle* h, void* stream) {
  if (!h) return MLP_ERR_INVALID_ARG;
  if (!h->shadow) return MLP_OK;
  return launch_shadow(h->params, h->shadow, buf_dtype(h), h->n_params, h->segs, S(stream));
}

mlp_status mlp_forward(mlp_handle* h, const void* x, int x_dtype, int batch, float* logits,
                       void* stream) {
  NvtxRange nvtx_range("mlp_forward");
  if (!h || batch < 0 || batch > h->max_batch) return MLP_ERR_INVALID_ARG;
  if (x_dtype != MLP_DTYPE_F32 && x_dtype != MLP_DTYPE_BF16 && x_dtype != MLP_DTYPE_U8 &&
      x_dtype != MLP_DTYPE_F16)
    return MLP_ERR_INVALID_ARG;
  if (batch == 0) return MLP_OK;
  if (!x || !logits) return MLP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(logits)) return MLP_ERR_MISALIGNED;
  cudaStream_t st = S(stream);
  MLP_CHECK(load_input(h, x, x_dtype, batch, st));
  MLP_CHECK(forward_hidden(h, batch, st));
  GemmArgs gl = logits_gemm(h, batch, logits, h->dims[h->L]);
  MLP_CHECK(run_gemm(with_simt_ws(h, gl), tc_prec(h->prec), st));
  h->have_forward = true;
  return MLP_OK;
}

mlp_status mlp_backward(mlp_handle* h, const void* dlogits, int ld_dlogits, int batch, void* dx,
                        void* stream) {
  NvtxRange nvtx_range("mlp_backward");
  if (!h || batch < 0 || batch > h->max_batch) return MLP_ERR_INVALID_ARG;
  if (batch == 0) return MLP_OK;
  if (!dlogits || !h->have_forward || ld_dlogits < h->dims[h->L]) return MLP_ERR_INVALID_ARG;
  if (!aligned16(dlogits) || (dx && !aligned16(dx))) return MLP_ERR_MISALIGNED;
  const bool bf = tc_prec(h->prec);
  if (bf && (ld_dlogits * 2) % 16 != 0) return MLP_ERR_MISALIGNED;
  return backward_impl(h, dlogits, ld_dlogits, batch, dx, false, 0.f, 0.f, S(stream));
}

mlp_status mlp_sgd_step(mlp_handle* h, float lr, float momentum, void* stream) {
  NvtxRange nvtx_range("mlp_sgd_step");
  if (!h) return MLP_ERR_INVALID_ARG;
  return launch_sgd(h->params, h->grads, h->velocity, h->shadow, buf_dtype(h), h->n_params, lr,
                    momentum, h->segs, S(stream));
}

mlp_status mlp_train_step(mlp_handle* h, const void* x, int x_dtype, const int32_t* labels,
                          int batch, float lr, float momentum, float* loss_out,
                          int32_t* argmax_out, void* stream) {
  NvtxRange nvtx_range("mlp_train_step");
  if (!h || batch < 0 || batch > h->max_batch) return MLP_ERR_INVALID_ARG;
  if (x_dtype != MLP_DTYPE_F32 && x_dtype != MLP_DTYPE_BF16 && x_dtype != MLP_DTYPE_U8 &&
      x_dtype != MLP_DTYPE_F16)
    return MLP_ERR_INVALID_ARG;
  if (batch == 0) return MLP_OK;
  if (!x || !labels) return MLP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(labels) || (loss_out && !aligned16(loss_out)) ||
      (argmax_out && !aligned16(argmax_out)))
    return MLP_ERR_MISALIGNED;
  return train_step_impl(h, x, x_dtype, labels, batch, lr, momentum, loss_out, argmax_out,
                         S(stream));
}

mlp_status mlp_train_epoch(mlp_handle* h, const void* x, int x_dtype, const int32_t* labels,
                           int n_samples, int batch, float lr, float momentum, float* losses_out,
                           int32_t* argmax_out, void* stream) {
  NvtxRange nvtx_range("mlp_train_epoch");
  if (!h || n_samples < 0 || batch <= 0 || batch > h->max_batch) return MLP_ERR_INVALID_ARG;
  if (x_dtype != MLP_DTYPE_F32 && x_dtype != MLP_DTYPE_BF16 && x_dtype != MLP_DTYPE_U8 &&
      x_dtype != MLP_DTYPE_F16)
    return MLP_ERR_INVALID_ARG;
  if (n_samples == 0) return MLP_OK;
  if (!x || !labels) return MLP_ERR_INVALID_ARG;
  const int xsz = x_dtype == MLP_DTYPE_U8 ? 1 : (x_dtype == MLP_DTYPE_F32 ? 4 : 2);
  const long long x_step = (long long)batch * h->dims[0] * xsz;
  // every step's input rows, labels and predictions start on 16 bytes
  if (!aligned16(x) || !aligned16(labels) || (argmax_out && !aligned16(argmax_out)) ||
      x_step % 16 != 0 || ((long long)batch * 4) % 16 != 0 ||
      (losses_out && (reinterpret_cast<uintptr_t>(losses_out) & 3)))
    return MLP_ERR_MISALIGNED;
  cudaStream_t st = S(stream);
  const int full = n_samples / batch, rem = n_samples % batch;
  int done = 0;
  if (full > 0) {
    StepSpec spec;
    float* loss = losses_out ? losses_out : h->loss;
    if (build_step_spec(h, x, x_dtype, labels, batch, lr, momentum, loss, argmax_out, st, &spec)) {
      spec.n_steps = full;
      spec.cast_stride = x_step;
      spec.label_stride = batch;
      spec.loss_stride = losses_out ? 1 : 0;
      spec.argmax_stride = batch;
      if (full > 1) spec.cast_dst_alt = h->x_copy_alt;
      MLP_CHECK(ensure_ones(h, st));
      MLP_CHECK(launch_step_program(spec, h->step_bar, wait_limit_ns(), st));
      // with two input buffers the last step (index full - 1) read the second
      // one when full is even: keep x_copy naming the latest input
      if (spec.cast_dst_alt && full % 2 == 0) std::swap(h->x_copy, h->x_copy_alt);
      h->have_forward = true;
      done = full;
    }
  }
  for (int s = done; s < full + (rem > 0 ? 1 : 0); ++s) {
    const int b = s < full ? batch : rem;
    MLP_CHECK(train_step_impl(h, static_cast<const uint8_t*>(x) + s * x_step, x_dtype,
                              labels + (size_t)s * batch, b, lr, momentum,
                              losses_out ? losses_out + s : nullptr,
                              argmax_out ? argmax_out + (size_t)s * batch : nullptr, st));
  }
  return MLP_OK;
}

}  // extern "C"
