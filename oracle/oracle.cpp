// Oracle for the MLP training step: plain, slow, double-precision CPU code.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
// its Python binding) links, imports or calls this file.  Only the tests, the
// package smoke check and the bench's CPU-baseline leg use it.  It shares no
// code, header, table or helper with the CUDA path.
//
// Every function is the plain definition of what it computes, written out with
// explicit loops in fp64 (summation in index order; OpenMP splits only
// independent outputs, never a sum), except the two linear-order functions,
// which state an exact sequence of fp32 operations.  Sources, by page and section:
//
//   [cap]  "Capstone 5: train a network with your CUDA kernels" (Day 100):
//          "The minimum model", "Work through the backward pass",
//          "Check your mapping", "Read the worked reference",
//          "Stage 2: backward and update".
//   [mk]   "Full-Depth MLP Megakernel + Fused Attention Preprocessing":
//          "What Worked" (RMSNorm -> gate -> LeakyReLU^2 -> down -> residual).
//   [vk]   "The Work Moved Down a Layer": "The Debugging Lesson Was Numerical"
//          (bf16/fp16 operands, fp32 accumulation, fp32 epilogue).
//   [hv]   "HIP + Vulkan backends -- Phase 3 (path to 100%)": "Vulkan /
//          SPIR-V", "Phase-3 bug hunt" (left-to-right sums for bit parity).
//
// Readings where the pages are silent (each also listed in the design notes):
//   * loss is the mean over the batch, so dZ carries 1/B;
//   * ReLU mask is (pre-activation > 0): a value at or below zero passes no
//     gradient ([cap] "Check your mapping");
//   * LeakyReLU^2: f(u) = u^2 for u > 0, (slope*u)^2 otherwise; the slope is a
//     parameter (0.5 in the block workloads);
//   * RMSNorm gain is the constant 1 and eps sits inside the square root;
//   * the blocks carry no biases;
//   * flat MLP parameter order W1, b1, W2, b2, ...; W_l is [in][out] row-major;
//   * flat stack parameter order per block: W_gate [d][h], then W_down [h][d];
//   * MSE is the mean over all T*d elements.
//
// Optional rounding-points modes round exactly where a tensor-core path stores
// a 16-bit operand: the input X, the weights, the stored hidden activation H,
// and the gradients dZ / dH fed to the backward matrix multiplies.  Everything
// else stays fp64.  points = 1 ("bf16 points") rounds to nearest-even with 8
// significant bits; points = 2 ("fp16 points", the FP16-operand choice of
// [vk]) rounds to the nearest IEEE binary16 value (11 significant bits,
// subnormals below 2^-14, overflow to infinity).  points = 0 is exact.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>
#include <omp.h>

extern "C" {

// Threads of the OpenMP loops below (timing runs only; results do not
// depend on it: every reduction sums in a fixed order within one thread).
void orc_set_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
int orc_max_threads() { return omp_get_max_threads(); }

// ---------------------------------------------------------------- helpers

// Round a double to the nearest value with 8 significant bits (the bf16
// significand), ties to even.  Used only in bf16-points mode.
double orc_round_bf16(double v) {
  if (v == 0.0 || !std::isfinite(v)) return v;
  int e = 0;
  double f = std::frexp(v, &e);             // v = f * 2^e, 0.5 <= |f| < 1
  double q = std::nearbyint(std::ldexp(f, 8));  // 8 significant bits
  return std::ldexp(q, e - 8);
}

// Round a double to the nearest IEEE 754 binary16 value, ties to even:
// 11 significant bits for |v| >= 2^-14 (the smallest normal), a fixed step of
// 2^-24 below it (subnormals), and +-infinity once the rounded magnitude
// exceeds the largest finite value 65504.  Used only in fp16-points mode.
double orc_round_f16(double v) {
  if (v == 0.0 || !std::isfinite(v)) return v;
  const double a = std::fabs(v);
  int e = 0;
  std::frexp(a, &e);                  // a = f * 2^e, 0.5 <= f < 1
  int step = e - 11;                  // exponent of the spacing at a
  if (step < -24) step = -24;         // subnormal spacing
  const double r = std::ldexp(std::nearbyint(std::ldexp(a, -step)), step);
  const double out = r > 65504.0 ? INFINITY : r;
  return std::copysign(out, v);
}

// points: 0 exact, 1 bf16, 2 fp16 (see the header comment).
static inline double maybe_round(double v, int points) {
  return points == 1 ? orc_round_bf16(v) : (points == 2 ? orc_round_f16(v) : v);
}

// [cap] "Predict the profile": the 784-256-10 network has 203,530 parameters;
// each layer holds an [in][out] weight and an [out] bias.
long long orc_param_count(const int* dims, int n_dims) {
  long long n = 0;
  for (int l = 0; l + 1 < n_dims; ++l)
    n += (long long)dims[l] * dims[l + 1] + dims[l + 1];
  return n;
}

// C[M][N] = sum_k A(m,k) * B(k,n).
//   a_t = 0: A stored [M][K];  a_t = 1: A stored [K][M]  (A is a transposed view)
//   b_t = 0: B stored [K][N];  b_t = 1: B stored [N][K]
// [cap] "Work through the backward pass": the weight and input gradients are
// matrix multiplies with one transposed input.
// Every entry is acc = 0; acc = acc + A(m,k) * B(k,n) for k = 0, 1, ..., K-1
// (each product and sum rounded to double, no contraction).  The loops visit
// entries in blocks of rows and columns so that a row of B is reused across
// several rows of C, but each entry still receives its K terms one at a time
// in ascending k, so the result is the same as the plain triple loop.
void orc_matmul(const double* A, int a_t, const double* B, int b_t,
                long long M, long long N, long long K, double* C) {
  constexpr long long MB = 8, NB = 256;
  // B as [K][N] rows (a plain copy of the transposed storage when b_t = 1)
  std::vector<double> Bt;
  const double* Bk = B;
  if (b_t) {
    Bt.resize((size_t)K * N);
    for (long long n = 0; n < N; ++n)
      for (long long k = 0; k < K; ++k) Bt[(size_t)k * N + n] = B[n * K + k];
    Bk = Bt.data();
  }
  const long long mblocks = (M + MB - 1) / MB, nblocks = (N + NB - 1) / NB;
#pragma omp parallel for schedule(dynamic, 1)
  for (long long blk = 0; blk < mblocks * nblocks; ++blk) {
    const long long m0 = (blk / nblocks) * MB, n0 = (blk % nblocks) * NB;
    const long long mr = std::min(MB, M - m0), nr = std::min(NB, N - n0);
    double acc[MB][NB];
    for (long long i = 0; i < mr; ++i)
      for (long long j = 0; j < nr; ++j) acc[i][j] = 0.0;
    for (long long k = 0; k < K; ++k) {
      const double* brow = Bk + k * N + n0;
      for (long long i = 0; i < mr; ++i) {
        const double a = a_t ? A[k * M + m0 + i] : A[(m0 + i) * K + k];
        double* ci = acc[i];
        for (long long j = 0; j < nr; ++j) ci[j] = ci[j] + a * brow[j];
      }
    }
    for (long long i = 0; i < mr; ++i)
      for (long long j = 0; j < nr; ++j) C[(m0 + i) * N + n0 + j] = acc[i][j];
  }
}

// Same definition, evaluated only at the listed (i, j) entries, from float
// storage (bf16 and fp32 values are exact in float).
void orc_matmul_entries_f32(const float* A, int a_t, const float* B, int b_t,
                            long long M, long long N, long long K,
                            const long long* ii, const long long* jj, long long n_entries,
                            double* out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (long long e = 0; e < n_entries; ++e) {
    long long m = ii[e], n = jj[e];
    double acc = 0.0;
    for (long long k = 0; k < K; ++k) {
      double a = a_t ? (double)A[k * M + m] : (double)A[m * K + k];
      double b = b_t ? (double)B[n * K + k] : (double)B[k * N + n];
      acc += a * b;
    }
    out[e] = acc;
  }
}

// ---------------------------------------------------------------- MLP

static long long weight_offset(const int* dims, int l) {
  long long off = 0;
  for (int i = 0; i < l; ++i) off += (long long)dims[i] * dims[i + 1] + dims[i + 1];
  return off;
}

// [cap] "The minimum model": H = ReLU(X W1 + b1), Z = H W2 + b2; every layer
// but the last applies ReLU (deeper MLPs repeat the hidden layer).
// acts receives H_1 .. H_{L-1} back to back, each [B][dims[l]].
void orc_mlp_forward(const int* dims, int n_dims, const double* params,
                     const double* X, long long B, int points,
                     double* acts, double* Z) {
  const int L = n_dims - 1;
  std::vector<double> in((size_t)B * dims[0]);
  for (size_t i = 0; i < in.size(); ++i) in[i] = maybe_round(X[i], points);
  long long act_off = 0;
  for (int l = 0; l < L; ++l) {
    const int fi = dims[l], fo = dims[l + 1];
    const double* W = params + weight_offset(dims, l);
    const double* b = W + (long long)fi * fo;
    std::vector<double> Wr((size_t)fi * fo);
    for (size_t i = 0; i < Wr.size(); ++i) Wr[i] = maybe_round(W[i], points);
    std::vector<double> out((size_t)B * fo);
    orc_matmul(in.data(), 0, Wr.data(), 0, B, fo, fi, out.data());
    const bool last = (l == L - 1);
    for (long long r = 0; r < B; ++r)
      for (int c = 0; c < fo; ++c) {
        double v = out[r * fo + c] + b[c];
        if (!last) v = maybe_round(v > 0.0 ? v : 0.0, points);
        out[r * fo + c] = v;
      }
    if (last) {
      std::memcpy(Z, out.data(), out.size() * sizeof(double));
    } else {
      std::memcpy(acts + act_off, out.data(), out.size() * sizeof(double));
      act_off += (long long)B * fo;
      in.swap(out);
    }
  }
}

// [cap] "The minimum model" and "Read the worked reference": stable softmax
// cross entropy.  Per row: m = max_c z, s = sum_c exp(z_c - m),
// loss_i = m + ln s - z_y; loss = mean over rows; p = exp(z - m) / s;
// dZ = (p - onehot(y)) / B.  argmax takes the lowest index among equal maxima.
// B_norm is the divisor used for the mean and for dZ (the batch size).
void orc_softmax_xent(const double* Z, const int* y, long long B, int C, long long B_norm,
                      double* loss_mean, double* row_loss, double* dZ, int* argmax) {
  double total = 0.0;
  for (long long r = 0; r < B; ++r) {
    const double* z = Z + r * C;
    double m = z[0];
    int am = 0;
    for (int c = 1; c < C; ++c)
      if (z[c] > m) { m = z[c]; am = c; }
    double s = 0.0;
    for (int c = 0; c < C; ++c) s += std::exp(z[c] - m);
    double li = m + std::log(s) - z[y[r]];
    if (row_loss) row_loss[r] = li;
    total += li;
    if (argmax) argmax[r] = am;
    if (dZ)
      for (int c = 0; c < C; ++c) {
        double p = std::exp(z[c] - m) / s;
        dZ[r * C + c] = (p - (c == y[r] ? 1.0 : 0.0)) / (double)B_norm;
      }
  }
  if (loss_mean) *loss_mean = total / (double)B_norm;
}

// [cap] "Work through the backward pass", layer by layer from the top:
//   dW_l = In_l^T dY_l,  db_l = sum_rows(dY_l),
//   dY_{l-1} = (dY_l W_l^T) * (H_l > 0),  dX = dY_0 W_0^T.
// grads has the flat parameter layout.  dX may be null.
void orc_mlp_backward(const int* dims, int n_dims, const double* params,
                      const double* X, long long B, const double* acts,
                      const double* dZ, int points, double* grads, double* dX) {
  const int L = n_dims - 1;
  std::vector<long long> act_off(L, 0);
  for (int l = 1; l < L; ++l) act_off[l] = (l == 1 ? 0 : act_off[l - 1] + B * dims[l - 1]);
  std::vector<double> dY((size_t)B * dims[L]);
  for (size_t i = 0; i < dY.size(); ++i) dY[i] = maybe_round(dZ[i], points);
  for (int l = L - 1; l >= 0; --l) {
    const int fi = dims[l], fo = dims[l + 1];
    const double* W = params + weight_offset(dims, l);
    double* dW = grads + weight_offset(dims, l);
    double* db = dW + (long long)fi * fo;
    std::vector<double> in((size_t)B * fi);
    if (l == 0) {
      for (size_t i = 0; i < in.size(); ++i) in[i] = maybe_round(X[i], points);
    } else {
      std::memcpy(in.data(), acts + act_off[l], in.size() * sizeof(double));
    }
    orc_matmul(in.data(), 1, dY.data(), 0, fi, fo, B, dW);
    for (int c = 0; c < fo; ++c) {
      double s = 0.0;
      for (long long r = 0; r < B; ++r) s += dY[r * fo + c];
      db[c] = s;
    }
    if (l == 0 && dX == nullptr) break;
    std::vector<double> Wr((size_t)fi * fo);
    for (size_t i = 0; i < Wr.size(); ++i) Wr[i] = maybe_round(W[i], points);
    std::vector<double> dIn((size_t)B * fi);
    orc_matmul(dY.data(), 0, Wr.data(), 1, B, fi, fo, dIn.data());
    if (l == 0) {
      std::memcpy(dX, dIn.data(), dIn.size() * sizeof(double));
      break;
    }
    const double* H = acts + act_off[l];
    for (size_t i = 0; i < dIn.size(); ++i)
      dIn[i] = maybe_round(H[i] > 0.0 ? dIn[i] : 0.0, points);
    dY.swap(dIn);
  }
}

// [cap] "Check your mapping": a bias gradient is a column reduction over the
// batch, out[c] = sum_r X[r][c] (rows in order).  X is float storage.
void orc_colsum_f32(const float* X, long long rows, long long cols, long long ld, double* out) {
  for (long long c = 0; c < cols; ++c) {
    double s = 0.0;
    for (long long r = 0; r < rows; ++r) s += (double)X[r * ld + c];
    out[c] = s;
  }
}

// ---------------------------------------------------------------- linear order
// The linear-order fp32 forms ([hv] "HIP + Vulkan backends -- Phase 3 (path
// to 100%)", "Vulkan / SPIR-V" and "Phase-3 bug hunt": sum left to right, one
// element after another, so that a device sum made in the same order agrees
// bit for bit).  These two are fp32 by definition, not fp64: they state the
// exact sequence of single-precision operations a linear-order sum performs.

// C[m][n] = act(chain + bias[n]) where chain = fma(a_{K-1}, b_{K-1}, ... fma(a_0,
// b_0, 0)), every step one correctly rounded single-precision fused
// multiply-add; bias (nullable) is one fp32 add; act 1 = ReLU (max with 0);
// mask (nullable, [M][ldm]) keeps C where mask > 0.  A is [M][K] (a_t = 0) or
// [K][M]; B is [K][N] (b_t = 0) or [N][K].
void orc_matmul_f32_linear(const float* A, int a_t, const float* B, int b_t, long long M,
                           long long N, long long K, const float* bias, int act,
                           const float* mask, long long ldm, float* C) {
#pragma omp parallel for schedule(static)
  for (long long m = 0; m < M; ++m) {
    for (long long n = 0; n < N; ++n) {
      float acc = 0.0f;
      for (long long k = 0; k < K; ++k) {
        const float a = a_t ? A[k * M + m] : A[m * K + k];
        const float b = b_t ? B[n * K + k] : B[k * N + n];
        acc = std::fma(a, b, acc);
      }
      float v = acc;
      if (bias) v = v + bias[n];
      if (act == 1) v = v > 0.0f ? v : 0.0f;
      if (mask && !(mask[m * ldm + n] > 0.0f)) v = 0.0f;
      C[m * N + n] = v;
    }
  }
}

// out[c] = ((X[0][c] + X[1][c]) + X[2][c]) + ... in fp32, starting from 0.
void orc_colsum_f32_linear(const float* X, long long rows, long long cols, long long ld,
                           float* out) {
  for (long long c = 0; c < cols; ++c) {
    float s = 0.0f;
    for (long long r = 0; r < rows; ++r) s = s + X[r * ld + c];
    out[c] = s;
  }
}

// [cap] "Read the worked reference": momentum SGD over one flat buffer,
// v <- momentum * v - lr * g;  w <- w + v.
void orc_sgd_momentum(double* w, const double* g, double* v, long long n,
                      double lr, double momentum) {
  for (long long i = 0; i < n; ++i) {
    v[i] = momentum * v[i] - lr * g[i];
    w[i] = w[i] + v[i];
  }
}

// One full training step (forward, loss, backward, update), composed from the
// functions above.  Returns the mean loss; grads (nullable) receives the flat
// gradient; acts/Z/dZ are internal.
double orc_mlp_train_step(const int* dims, int n_dims, double* params, double* velocity,
                          const double* X, const int* y, long long B, double lr,
                          double momentum, int points, double* grads_out) {
  const int L = n_dims - 1;
  long long n_act = 0;
  for (int l = 1; l < L; ++l) n_act += B * dims[l];
  std::vector<double> acts((size_t)std::max<long long>(n_act, 1));
  std::vector<double> Z((size_t)B * dims[L]), dZ((size_t)B * dims[L]);
  orc_mlp_forward(dims, n_dims, params, X, B, points, acts.data(), Z.data());
  double loss = 0.0;
  orc_softmax_xent(Z.data(), y, B, dims[L], B, &loss, nullptr, dZ.data(), nullptr);
  const long long P = orc_param_count(dims, n_dims);
  std::vector<double> g((size_t)P);
  orc_mlp_backward(dims, n_dims, params, X, B, acts.data(), dZ.data(), points,
                   g.data(), nullptr);
  if (grads_out) std::memcpy(grads_out, g.data(), (size_t)P * sizeof(double));
  orc_sgd_momentum(params, g.data(), velocity, P, lr, momentum);
  return loss;
}

// Row-separable forward on float storage: logits (and optionally the hidden
// activations of the listed rows) for selected rows of a large batch.
void orc_mlp_forward_rows_f32(const int* dims, int n_dims, const float* params,
                              const float* X, const long long* rows, long long n_rows,
                              int points, double* Z_rows) {
  const int L = n_dims - 1;
#pragma omp parallel for schedule(dynamic, 1)
  for (long long e = 0; e < n_rows; ++e) {
    std::vector<double> in(dims[0]);
    for (int i = 0; i < dims[0]; ++i)
      in[i] = maybe_round((double)X[rows[e] * dims[0] + i], points);
    for (int l = 0; l < L; ++l) {
      const int fi = dims[l], fo = dims[l + 1];
      const float* W = params + weight_offset(dims, l);
      const float* b = W + (long long)fi * fo;
      std::vector<double> out(fo, 0.0);
      for (int c = 0; c < fo; ++c) {
        double acc = 0.0;
        for (int k = 0; k < fi; ++k) acc += in[k] * maybe_round((double)W[(long long)k * fo + c], points);
        out[c] = acc + (double)b[c];
      }
      if (l < L - 1)
        for (int c = 0; c < fo; ++c) out[c] = maybe_round(out[c] > 0.0 ? out[c] : 0.0, points);
      in.swap(out);
    }
    for (int c = 0; c < dims[L]; ++c) Z_rows[e * dims[L] + c] = in[c];
  }
}

// ---------------------------------------------------------------- MLP block

// LeakyReLU^2 and its derivative ([mk] "What Worked").  f(u) = u^2 for u > 0,
// (slope u)^2 otherwise; f'(u) = 2u for u > 0, 2 slope^2 u otherwise (0 at 0).
static inline double lrelu_sq(double u, double slope) {
  double t = u > 0.0 ? u : slope * u;
  return t * t;
}
static inline double lrelu_sq_grad(double u, double slope) {
  return u > 0.0 ? 2.0 * u : 2.0 * slope * slope * u;
}

// RMSNorm with gain 1: r = 1 / sqrt(mean(x^2) + eps), n = x r.
static inline double rms_rstd(const double* x, int d, double eps) {
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += x[i] * x[i];
  return 1.0 / std::sqrt(ss / (double)d + eps);
}

// One token of the block forward:
//   n = RMSNorm(x); u = n W_gate; a = LeakyReLU^2(u); y = x + a W_down.
static void block_fwd_token(const double* x, const double* Wg, const double* Wd,
                            int d, int h, double eps, double slope,
                            double* y, double* rstd, double* u_out, double* a_out) {
  const double r = rms_rstd(x, d, eps);
  std::vector<double> n(d), u(h, 0.0), a(h), z(d, 0.0);
  for (int i = 0; i < d; ++i) n[i] = x[i] * r;
  // u_j = sum_i n_i Wg[i][j], each u_j summing over ascending i from 0 (the
  // loops run over i outside so that rows of W_gate are read in order)
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < h; ++j) u[j] = u[j] + n[i] * Wg[(long long)i * h + j];
  for (int j = 0; j < h; ++j) a[j] = lrelu_sq(u[j], slope);
  // z_i = sum_j a_j Wd[j][i] over ascending j, then y = x + z
  for (int j = 0; j < h; ++j)
    for (int i = 0; i < d; ++i) z[i] = z[i] + a[j] * Wd[(long long)j * d + i];
  for (int i = 0; i < d; ++i) y[i] = x[i] + z[i];
  if (rstd) *rstd = r;
  if (u_out) std::memcpy(u_out, u.data(), h * sizeof(double));
  if (a_out) std::memcpy(a_out, a.data(), h * sizeof(double));
}

// [mk] "What Worked": y = x + LeakyReLU^2(RMSNorm(x) W_gate) W_down, per token.
void orc_block_fwd(const double* x, const double* Wg, const double* Wd, long long T,
                   int d, int h, double eps, double slope, double* y, double* rstd) {
#pragma omp parallel for schedule(static)
  for (long long t = 0; t < T; ++t)
    block_fwd_token(x + t * d, Wg, Wd, d, h, eps, slope, y + t * d,
                    rstd ? rstd + t : nullptr, nullptr, nullptr);
}

// Backward of one token, given upstream dy; accumulates nothing (returns the
// per-token pieces):  da = dy W_down^T;  du = da * f'(u);
// dn = du W_gate^T;  dx = dy + r (dn - n mean(dn * n)).
static void block_bwd_token(const double* x, const double* Wg, const double* Wd,
                            const double* dy, int d, int h, double eps, double slope,
                            double* dx, double* n_out, double* a_out, double* du_out) {
  double r = 0.0;
  std::vector<double> u(h), a(h), n(d), du(h);
  block_fwd_token(x, Wg, Wd, d, h, eps, slope, dx /*scratch*/, &r, u.data(), a.data());
  for (int i = 0; i < d; ++i) n[i] = x[i] * r;
  for (int j = 0; j < h; ++j) {
    double da = 0.0;
    for (int i = 0; i < d; ++i) da += dy[i] * Wd[(long long)j * d + i];
    du[j] = da * lrelu_sq_grad(u[j], slope);
  }
  std::vector<double> dn(d);
  double dot = 0.0;
  for (int i = 0; i < d; ++i) {
    double acc = 0.0;
    for (int j = 0; j < h; ++j) acc += du[j] * Wg[(long long)i * h + j];
    dn[i] = acc;
    dot += acc * n[i];
  }
  const double mean_dn_n = dot / (double)d;
  for (int i = 0; i < d; ++i) dx[i] = dy[i] + r * (dn[i] - n[i] * mean_dn_n);
  if (n_out) std::memcpy(n_out, n.data(), d * sizeof(double));
  if (a_out) std::memcpy(a_out, a.data(), h * sizeof(double));
  if (du_out) std::memcpy(du_out, du.data(), h * sizeof(double));
}

// Full block backward: dx per token; dW_down = A^T dY and dW_gate = N^T dU
// summed over all tokens (token order).
void orc_block_bwd(const double* x, const double* Wg, const double* Wd, const double* dy,
                   long long T, int d, int h, double eps, double slope,
                   double* dx, double* dWg, double* dWd) {
  std::vector<double> N((size_t)T * d), A((size_t)T * h), DU((size_t)T * h);
#pragma omp parallel for schedule(static)
  for (long long t = 0; t < T; ++t)
    block_bwd_token(x + t * d, Wg, Wd, dy + t * d, d, h, eps, slope, dx + t * d,
                    N.data() + t * d, A.data() + t * h, DU.data() + t * h);
  orc_matmul(A.data(), 1, dy, 0, h, d, T, dWd);
  orc_matmul(N.data(), 1, DU.data(), 0, d, h, T, dWg);
}

// Sampled forms on float storage (row-separable outputs).
void orc_block_fwd_rows_f32(const float* x, const float* Wg, const float* Wd, int d, int h,
                            double eps, double slope, const long long* rows, long long n_rows,
                            double* y, double* rstd) {
  std::vector<double> wg((size_t)d * h), wd((size_t)h * d);
  for (size_t i = 0; i < wg.size(); ++i) wg[i] = Wg[i];
  for (size_t i = 0; i < wd.size(); ++i) wd[i] = Wd[i];
#pragma omp parallel for schedule(dynamic, 4)
  for (long long e = 0; e < n_rows; ++e) {
    std::vector<double> xr(d);
    for (int i = 0; i < d; ++i) xr[i] = x[rows[e] * d + i];
    block_fwd_token(xr.data(), wg.data(), wd.data(), d, h, eps, slope, y + e * d,
                    rstd ? rstd + e : nullptr, nullptr, nullptr);
  }
}

void orc_block_bwd_dx_rows_f32(const float* x, const float* Wg, const float* Wd, const float* dy,
                               int d, int h, double eps, double slope,
                               const long long* rows, long long n_rows, double* dx) {
  std::vector<double> wg((size_t)d * h), wd((size_t)h * d);
  for (size_t i = 0; i < wg.size(); ++i) wg[i] = Wg[i];
  for (size_t i = 0; i < wd.size(); ++i) wd[i] = Wd[i];
#pragma omp parallel for schedule(dynamic, 4)
  for (long long e = 0; e < n_rows; ++e) {
    std::vector<double> xr(d), dyr(d);
    for (int i = 0; i < d; ++i) { xr[i] = x[rows[e] * d + i]; dyr[i] = dy[rows[e] * d + i]; }
    block_bwd_token(xr.data(), wg.data(), wd.data(), dyr.data(), d, h, eps, slope,
                    dx + e * d, nullptr, nullptr, nullptr);
  }
}

// Selected weight-gradient entries: which = 0 -> dW_gate[i][j] = sum_t n_ti du_tj,
// which = 1 -> dW_down[i][j] = sum_t a_ti dy_tj.  Each entry sums over all T
// tokens in token order.
void orc_block_bwd_dw_entries_f32(const float* x, const float* Wg, const float* Wd,
                                  const float* dy, long long T, int d, int h, double eps,
                                  double slope, const int* which, const long long* ii,
                                  const long long* jj, long long n_entries, double* out) {
  std::vector<double> r((size_t)T);
#pragma omp parallel for schedule(static)
  for (long long t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int i = 0; i < d; ++i) { double v = x[t * d + i]; ss += v * v; }
    r[t] = 1.0 / std::sqrt(ss / (double)d + eps);
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (long long e = 0; e < n_entries; ++e) {
    double acc = 0.0;
    if (which[e] == 1) {  // dW_down[j_hidden = ii][i_model = jj]
      const long long jh = ii[e], im = jj[e];
      for (long long t = 0; t < T; ++t) {
        double u = 0.0;
        for (int k = 0; k < d; ++k) u += (double)x[t * d + k] * r[t] * (double)Wg[(long long)k * h + jh];
        acc += lrelu_sq(u, slope) * (double)dy[t * d + im];
      }
    } else {              // dW_gate[i_model = ii][j_hidden = jj]
      const long long im = ii[e], jh = jj[e];
      for (long long t = 0; t < T; ++t) {
        double u = 0.0, da = 0.0;
        for (int k = 0; k < d; ++k) {
          u += (double)x[t * d + k] * r[t] * (double)Wg[(long long)k * h + jh];
          da += (double)dy[t * d + k] * (double)Wd[jh * d + k];
        }
        const double du = da * lrelu_sq_grad(u, slope);
        acc += (double)x[t * d + im] * r[t] * du;
      }
    }
    out[e] = acc;
  }
}

// Mean-squared loss: L = mean((y - t)^2) over n elements; dy = 2 (y - t) / n.
void orc_mse(const double* y, const double* t, long long n, double* loss, double* dy) {
  double s = 0.0;
  for (long long i = 0; i < n; ++i) {
    double e = y[i] - t[i];
    s += e * e;
    if (dy) dy[i] = 2.0 * e / (double)n;
  }
  if (loss) *loss = s / (double)n;
}

// A stack of blocks with the mean-squared loss on the last output, then the
// backward through all blocks.  params: per block W_gate [d][h] then
// W_down [h][d].  grads has the same layout.  Returns the loss.
double orc_stack_fwd_bwd(const double* x0, const double* params, int n_blocks, long long T,
                         int d, int h, double eps, double slope, const double* target,
                         double* grads, double* dx0) {
  const long long per = 2LL * d * h;
  std::vector<std::vector<double>> xs(n_blocks + 1, std::vector<double>((size_t)T * d));
  std::memcpy(xs[0].data(), x0, (size_t)T * d * sizeof(double));
  for (int b = 0; b < n_blocks; ++b)
    orc_block_fwd(xs[b].data(), params + b * per, params + b * per + (long long)d * h, T, d, h,
                  eps, slope, xs[b + 1].data(), nullptr);
  double loss = 0.0;
  std::vector<double> dy((size_t)T * d), dx((size_t)T * d);
  orc_mse(xs[n_blocks].data(), target, T * d, &loss, dy.data());
  for (int b = n_blocks - 1; b >= 0; --b) {
    orc_block_bwd(xs[b].data(), params + b * per, params + b * per + (long long)d * h, dy.data(),
                  T, d, h, eps, slope, dx.data(), grads + b * per,
                  grads + b * per + (long long)d * h);
    dy.swap(dx);
  }
  if (dx0) std::memcpy(dx0, dy.data(), (size_t)T * d * sizeof(double));
  return loss;
}

// ---------------------------------------------------------------- attention prep
// [mk] "What Worked" (attention preprocessing fusion) and "What Didn't Work"
// (the fully fused form: RMSNorm -> QKV projection -> QK norm -> RoPE -> gain,
// achievable in raw CUDA).  Per token t at position p = t mod seq_len:
//   r = 1 / sqrt(mean_i x_i^2 + eps);  u = r (x W_qkv)      (RMSNorm, gain 1)
//   u splits into n_q query heads, n_kv key heads, n_kv value heads of hd;
//   query and key heads:  u_h <- u_h / sqrt(mean_j u_hj^2 + eps)   (QK norm)
//                         partial RoPE on dims [0, R): for i < R/2,
//                           a = p theta^(-2i/R),
//                           (u_i, u_{i+R/2}) <- (u_i cos a - u_{i+R/2} sin a,
//                                                u_{i+R/2} cos a + u_i sin a)
//   query heads:          u_h <- q_gain[h] u_h
//   value heads:          unchanged.
// x [T][d], W [d][N] with N = (n_q + 2 n_kv) hd, out [T][N].
static void attn_prep_token(const double* x, const double* W, const double* q_gain, int d,
                            int n_q, int n_kv, int hd, int R, long long pos, double eps,
                            double theta, double* out) {
  const int N = (n_q + 2 * n_kv) * hd;
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += x[i] * x[i];
  const double r = 1.0 / std::sqrt(ss / d + eps);
  for (int n = 0; n < N; ++n) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i) acc += x[i] * W[(long long)i * N + n];
    out[n] = r * acc;
  }
  for (int h = 0; h < n_q + n_kv; ++h) {
    double* u = out + (long long)h * hd;
    double hs = 0.0;
    for (int j = 0; j < hd; ++j) hs += u[j] * u[j];
    const double inv = 1.0 / std::sqrt(hs / hd + eps);
    for (int j = 0; j < hd; ++j) u[j] *= inv;
    for (int i = 0; i < R / 2; ++i) {
      const double a = (double)pos * std::pow(theta, -2.0 * i / R);
      const double c = std::cos(a), s = std::sin(a);
      const double x1 = u[i], x2 = u[i + R / 2];
      u[i] = x1 * c - x2 * s;
      u[i + R / 2] = x2 * c + x1 * s;
    }
    if (h < n_q)
      for (int j = 0; j < hd; ++j) u[j] *= q_gain[h];
  }
}

void orc_attn_prep(const double* x, const double* W, const double* q_gain, long long T, int d,
                   int n_q, int n_kv, int hd, int R, long long seq_len, double eps,
                   double theta, double* out) {
  const int N = (n_q + 2 * n_kv) * hd;
#pragma omp parallel for schedule(static)
  for (long long t = 0; t < T; ++t)
    attn_prep_token(x + t * d, W, q_gain, d, n_q, n_kv, hd, R, t % seq_len, eps, theta,
                    out + t * N);
}

// The same for the listed tokens only (x and W in fp32, as stored; outputs
// fp64), for spot checks of large problems.
void orc_attn_prep_rows_f32(const float* x, const float* W, const float* q_gain, int d, int n_q,
                            int n_kv, int hd, int R, long long seq_len, double eps,
                            double theta, const long long* rows, long long n_rows,
                            double* out) {
  const int N = (n_q + 2 * n_kv) * hd;
  std::vector<double> Wd((size_t)d * N), g(n_q > 0 ? n_q : 1);
  for (size_t i = 0; i < Wd.size(); ++i) Wd[i] = W[i];
  for (int h = 0; h < n_q; ++h) g[h] = q_gain[h];
#pragma omp parallel for schedule(dynamic, 1)
  for (long long e = 0; e < n_rows; ++e) {
    std::vector<double> xr(d);
    for (int i = 0; i < d; ++i) xr[i] = x[rows[e] * d + i];
    attn_prep_token(xr.data(), Wd.data(), g.data(), d, n_q, n_kv, hd, R, rows[e] % seq_len, eps,
                    theta, out + e * N);
  }
}

}  // extern "C"
