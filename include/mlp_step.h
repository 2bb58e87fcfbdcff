/*
 * mlp_step.h -- C ABI of the GB300 (sm_103a) MLP training-step library.
 *
 * One full MLP training step on one GPU: forward GEMMs with a fused bias and
 * activation epilogue, stable softmax cross entropy producing the loss and
 * dZ, the backward GEMMs with a transposed operand and the fused ReLU mask,
 * column-reduction bias gradients, and a flat-buffer momentum-SGD update; plus
 * the transformer MLP block (RMSNorm -> gate projection -> LeakyReLU^2 -> down
 * projection -> residual) forward and backward, a mean-squared loss, and a
 * stack of blocks.
 *
 * Sources (page title, section):
 *   [cap] "Capstone 5: train a network with your CUDA kernels" -- "The minimum
 *         model", "Work through the backward pass", "Check your mapping",
 *         "Read the worked reference", "Stage 2: backward and update".
 *   [mk]  "Full-Depth MLP Megakernel + Fused Attention Preprocessing" --
 *         "What Worked", "What Didn't Work".
 *   [vk]  "The Work Moved Down a Layer" -- "Cooperation Beats Isolation",
 *         "Keep state resident", "The Debugging Lesson Was Numerical".
 *   [hv]  "HIP + Vulkan backends -- Phase 3 (path to 100%)" -- "Vulkan /
 *         SPIR-V", "Phase-3 bug hunt" (linear-order sums for bit parity
 *         with a CPU oracle).
 *
 * Conventions for every call:
 *   - All tensors are caller-owned DEVICE memory (the library allocates
 *     nothing), row-major and contiguous along the last dimension, with the
 *     leading dimension given where one is taken.  Base pointers must be
 *     16-byte aligned (MLP_ERR_MISALIGNED otherwise); leading dimensions of
 *     bf16 / fp16 operands of the tensor-core path must make rows 16-byte
 *     aligned.
 *   - Weights are [in][out] (the X * W orientation of [cap] "The minimum
 *     model").  bf16 means bfloat16 rounded to nearest even from fp32, fp16
 *     IEEE binary16 rounded to nearest even.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work: no host synchronisation, no allocation, no host copies, so
 *     a whole step can be captured into a CUDA graph.
 *   - Errors are returned, never thrown.  Argument checks happen on the host
 *     before anything is enqueued; a failed check enqueues nothing.  A kernel
 *     that gives up on a bounded wait records the fact on the device;
 *     mlp_get_device_status() reports it as MLP_ERR_DEVICE_TIMEOUT.
 *   - Empty work (batch 0, n 0, M, N or T 0) returns MLP_OK and launches nothing.
 *   - There is no CPU fallback: every computation runs in this library's
 *     CUDA kernels on the current device.
 */
#ifndef MLP_STEP_H
#define MLP_STEP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int mlp_status;
#define MLP_OK 0
#define MLP_ERR_INVALID_ARG 1        /* null pointer, negative size, unknown enum   */
#define MLP_ERR_MISALIGNED 2         /* pointer or leading dimension not 16-B aligned */
#define MLP_ERR_UNSUPPORTED_SHAPE 3  /* a dimension outside what the kernels handle */
#define MLP_ERR_CUDA 4               /* a CUDA runtime call or launch failed        */
#define MLP_ERR_DEVICE_TIMEOUT 5     /* a kernel abandoned a bounded wait           */
#define MLP_ERR_NUMERIC 6            /* a loss kernel produced a non-finite loss    */

#define MLP_ACT_NONE 0
#define MLP_ACT_RELU 1               /* [cap] "The minimum model"                    */
#define MLP_ACT_LEAKY_RELU_SQ 2      /* [mk] "What Worked": (leaky_relu(u))^2        */

#define MLP_PREC_FP32 0              /* fp32 operands, fp32 SIMT kernels             */
#define MLP_PREC_BF16 1              /* bf16 operands, fp32 accumulation in tensor
                                        memory, fp32 epilogue ([vk] "The Debugging
                                        Lesson Was Numerical"), fp32 master weights  */
#define MLP_PREC_FP16 2              /* the same tensor-core path with fp16 operands
                                        (the FP16-in / FP32-accumulate choice of [vk]
                                        "The Debugging Lesson Was Numerical"): fp16
                                        input copy, weight shadow, hidden
                                        activations and gradients fed to the GEMMs */

#define MLP_DTYPE_F32 0
#define MLP_DTYPE_BF16 1
#define MLP_DTYPE_U8 2               /* image bytes; the value used is byte / 255    */
#define MLP_DTYPE_F16 3              /* IEEE binary16                                */

typedef struct mlp_handle mlp_handle;

/* Text for a status code.  Never NULL. */
const char* mlp_status_string(mlp_status s);

/* Synchronises `stream`, then reads and clears the device error word.
 * Returns MLP_ERR_DEVICE_TIMEOUT if a kernel abandoned a bounded wait since the
 * last call, MLP_ERR_NUMERIC if a loss computed since the last call (softmax
 * cross entropy, mean-squared loss, or the loss inside a training step) was
 * not finite ([cap] "The independent submission gate": a run that exits
 * cleanly is not yet a correct one), MLP_ERR_CUDA if the stream reports an
 * error, else MLP_OK.  The first event recorded since the last call wins. */
mlp_status mlp_get_device_status(void* stream);

/* Sets the time limit of every bounded wait in the kernels, in nanoseconds of
 * the GPU's global timer (0 restores the default of 2 s, far above any
 * legitimate wait).  Host-side setting, passed to kernels at launch. */
void mlp_set_wait_limit_ns(long long ns);

/* Summation order of the fp32 reductions that the library controls (the
 * linear-order sums of [hv] "Vulkan / SPIR-V" and "Phase-3 bug hunt": a
 * fixed, plain left-to-right order, so that a CPU loop summing the same way
 * reproduces the result bit for bit).
 *   MLP_ORDER_FAST (default): fp32 SIMT GEMMs may split K over CTAs (partial
 *     sums added in split order) and column sums reduce in chunks and trees;
 *     results are deterministic run to run.
 *   MLP_ORDER_LINEAR: every fp32 SIMT GEMM output is ONE fused-multiply-add
 *     chain over k = 0, 1, ..., K-1 starting from 0, then + bias (one fp32
 *     add), then the activation and mask; every column sum adds the rows
 *     r = 0, 1, ... into one fp32 accumulator starting from 0.  Slower (no
 *     split-K, one thread per column).
 * The tensor-core MMAs accumulate in the hardware's order in either mode, and
 * the loss uses IEEE exp and log; neither is covered.  Host-side setting,
 * read at each launch. */
#define MLP_ORDER_FAST 0
#define MLP_ORDER_LINEAR 1
mlp_status mlp_set_reduction_order(int order);
int mlp_get_reduction_order(void);

/* Self-test of the bounded-wait mechanism: launches one block that waits on a
 * shared-memory barrier nothing arrives at, for `limit_ns` nanoseconds, then
 * records MLP_ERR_DEVICE_TIMEOUT in the device error word and exits cleanly.
 * Read the result with mlp_get_device_status(). */
mlp_status mlp_selftest_wait_timeout(long long limit_ns, void* stream);

/* Number of kernels this library has enqueued (or recorded into a stream
 * capture) since it was loaded.  Host-side counter. */
unsigned long long mlp_launch_count(void);

/* Per-kernel timing for measurement: while enabled, every kernel launched on a
 * stream that is not being captured is bracketed by CUDA events on that
 * stream.  Enabling clears earlier records. */
mlp_status mlp_timing_enable(int on);

/* Synchronises the recorded events and writes a JSON object
 * {"kernel[shape]": [launches, total_ms], ...} into buf (truncated to cap-1
 * bytes, NUL-terminated).  Returns the bytes the full text needs. */
size_t mlp_timing_report(char* buf, size_t cap);

/* ---------------------------------------------------------------- MLP ------
 * An MLP with layer widths dims[0..n_dims-1]; every layer but the last applies
 * the hidden activation ([cap] "The minimum model": H = ReLU(X W1 + b1),
 * Z = H W2 + b2; deeper MLPs repeat the hidden layer).
 */

/* Number of fp32 parameters: sum over layers of in*out + out.  784-256-10
 * gives 203,530 ([cap] "Predict the profile").  Flat order W1, b1, W2, b2, ...
 * ([cap] "Read the worked reference": one flat buffer for all four tensors). */
size_t mlp_param_count(const int* dims, int n_dims);

/* Offset (in floats) of layer `layer`'s weight (which = 0) or bias (which = 1)
 * inside the flat buffer.  Returns (size_t)-1 for a bad layer or which. */
size_t mlp_param_offset(const int* dims, int n_dims, int layer, int which);

/* Elements of the 16-bit weight shadow used by MLP_PREC_BF16 (bf16) and
 * MLP_PREC_FP16 (fp16): each W_l stored
 * [in][out_pad] with out_pad = out rounded up to a multiple of 8 when out <= 16
 * (16-byte rows), else to a multiple of 64 (whole 128-byte lines, which the
 * tensor-core tiles read fastest), layers back to back.  Biases have no shadow
 * (the epilogue reads the fp32 bias). */
size_t mlp_shadow_elems(const int* dims, int n_dims);

/* Bytes of device workspace mlp_create needs for batches up to max_batch. */
size_t mlp_workspace_bytes(const int* dims, int n_dims, int max_batch, int prec);

/* Builds a host-side handle over caller-owned device buffers.
 *   params, velocity, grads: fp32[mlp_param_count], flat layout above.
 *   params_bf16: the 16-bit weight shadow, 16-byte aligned:
 *   bf16[mlp_shadow_elems] for MLP_PREC_BF16, fp16[mlp_shadow_elems] for
 *   MLP_PREC_FP16, NULL for MLP_PREC_FP32.
 *   workspace: ws_bytes >= mlp_workspace_bytes(...), holds saved activations,
 *   dZ/dH buffers and reduction partials between calls.
 *   hidden_act: MLP_ACT_RELU or MLP_ACT_NONE.
 * Nothing is launched.  The handle keeps pointers, never ownership.  One
 * handle serves one stream at a time.
 * Errors: INVALID_ARG (null, n_dims < 2, dims <= 0, max_batch <= 0,
 * ws_bytes too small), MISALIGNED. */
mlp_status mlp_create(const int* dims, int n_dims, int hidden_act, int prec, int max_batch,
                      float* params, float* velocity, float* grads, void* params_bf16,
                      void* workspace, size_t ws_bytes, mlp_handle** out);

/* Frees the host-side handle only. */
void mlp_destroy(mlp_handle* h);

/* Rewrites the 16-bit shadow from the fp32 parameters (after the caller
 * changed them).  No-op for MLP_PREC_FP32. */
mlp_status mlp_refresh_shadow(mlp_handle* h, void* stream);

/* Forward of `batch` rows of x ([batch][dims[0]], dtype x_dtype: F32, BF16,
 * F16 or U8; converted to the network's operand type).  Writes logits fp32 [batch][dims[-1]] and keeps the input copy and the
 * hidden activations in the workspace for mlp_backward.
 * ([cap] "The minimum model"; bias and ReLU live in the GEMM epilogue per
 * [cap] "Read the worked reference".)  batch <= max_batch. */
mlp_status mlp_forward(mlp_handle* h, const void* x, int x_dtype, int batch, float* logits,
                       void* stream);

/* Backward of the last mlp_forward, given dlogits = dL/dZ:
 *   dW_l = In_l^T dY_l,  db_l = sum_rows dY_l,  dY_{l-1} = (dY_l W_l^T) * (H_l > 0)
 * ([cap] "Work through the backward pass", "Check your mapping").
 * dlogits: [batch][ld_dlogits], fp32 for MLP_PREC_FP32, bf16 for MLP_PREC_BF16,
 * fp16 for MLP_PREC_FP16 (for 16-bit, ld_dlogits * 2 must be a multiple of 16).
 * Overwrites the handle's grads (no accumulation).  dx (nullable): [batch][dims[0]]
 * in the same type as dlogits, receives dX = dY_0 W_1^T. */
mlp_status mlp_backward(mlp_handle* h, const void* dlogits, int ld_dlogits, int batch, void* dx,
                        void* stream);

/* Momentum SGD over the handle's flat buffers, then (BF16, FP16) the shadow
 * refresh, in one kernel. */
mlp_status mlp_sgd_step(mlp_handle* h, float lr, float momentum, void* stream);

/* One full training step on the stream: forward, softmax cross entropy
 * (mean over the batch), backward, momentum SGD.  labels int32[batch] in
 * [0, dims[-1]).  loss_out (nullable): device fp32 scalar.  argmax_out
 * (nullable): device int32[batch] predictions of this step's forward.
 * For MLP_PREC_BF16 and MLP_PREC_FP16 networks with batch <= 128, at most 32
 * classes and small
 * layers (every GEMM of the step fits one round of CTAs and every weight
 * update rides in its gradient GEMM) the step is ONE cooperative kernel
 * launch whose phases are separated by grid barriers; results are the same
 * as with one launch per GEMM ([cap] "Capstone 5: train a network with your
 * CUDA kernels": the training loop of the minimum model). */
mlp_status mlp_train_step(mlp_handle* h, const void* x, int x_dtype, const int32_t* labels,
                          int batch, float lr, float momentum, float* loss_out,
                          int32_t* argmax_out, void* stream);

/* One epoch of training steps in sequence ([cap] "The minimum model": the
 * data set is visited in order in mini-batches): step s takes rows
 * [s * batch, min(n_samples, (s + 1) * batch)) of x ([n_samples][dims[0]],
 * dtype x_dtype) and of labels (int32[n_samples]); the last step takes the
 * remainder.  losses_out (nullable): device fp32[ceil(n_samples / batch)],
 * the mean loss of each step, 4-byte aligned.  argmax_out (nullable): device
 * int32[n_samples] predictions.  Exactly the results of calling
 * mlp_train_step on each step's slices in order; where a step is one
 * cooperative launch (see mlp_train_step) all full-size steps run in ONE
 * launch with a grid barrier between steps.  Each step's slice of x,
 * labels and argmax_out must start on 16 bytes (batch * dims[0] * element
 * size and batch * 4 multiples of 16, base pointers 16-byte aligned), else
 * MLP_ERR_MISALIGNED.  batch in [1, max_batch]. */
mlp_status mlp_train_epoch(mlp_handle* h, const void* x, int x_dtype, const int32_t* labels,
                           int n_samples, int batch, float lr, float momentum, float* losses_out,
                           int32_t* argmax_out, void* stream);

/* ---------------------------------------------------------------- loss -----
 * Stable softmax cross entropy, forward and backward ([cap] "The minimum
 * model", "Read the worked reference": subtract each row's maximum before
 * exponentiating; [vk]: fp32 reductions).  Per row i:
 *   m = max_c z_c,  s = sum_c exp(z_c - m),  loss_i = m + ln s - z_{y_i},
 *   dZ_ic = (exp(z_c - m) / s - [c == y_i]) / batch.
 * loss_out: device fp32 scalar = mean_i loss_i (fixed-order reduction, so the
 * result is bitwise reproducible).  logits fp32 [batch][ld_logits];
 * dlogits (nullable) [batch][ld_dlogits] fp32, bf16 or fp16 (dlogits_dtype); when
 * ld_dlogits > classes the padding columns are written as zero.  argmax_out
 * (nullable) int32[batch]: lowest index among equal maxima.
 * workspace: softmax_xent_workspace_bytes(batch, classes) bytes of scratch.
 * Labels outside [0, classes) are not checked on the device (the host cannot
 * see them); they give an unspecified loss for that row but no memory error. */
size_t softmax_xent_workspace_bytes(int batch, int classes);
mlp_status softmax_xent_fwd_bwd(const float* logits, int ld_logits, const int32_t* labels,
                                int batch, int classes, float* loss_out, void* dlogits,
                                int dlogits_dtype, int ld_dlogits, int32_t* argmax_out,
                                void* workspace, size_t ws_bytes, void* stream);

/* softmax_xent_fwd_bwd without a workspace argument, for callers that cannot
 * allocate device memory: code that runs inside a host framework owning the
 * whole device heap, a memory-pool or allocator callback, or a runtime that
 * forbids allocation after start-up.  The pages have no counterpart; this is a
 * deployment variant of the loss entry point above, with the same arguments
 * and results apart from the workspace.
 * Its scratch (the fixed-order partial sums of the batch mean) is a
 * file-scope device array of 65,536 floats (256 KiB) that every GPU which
 * loads the library holds until the process exits; batches above
 * softmax_xent_noalloc_max_batch() = 524,288 rows return
 * MLP_ERR_UNSUPPORTED_SHAPE.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current and keeps it
 * for the life of the process (a device reset invalidates it); make that
 * first call before any stream capture on the device.  The call allocates
 * nothing.  All calls share the one array and it keeps the last call's
 * contents (each call writes every partial it reads, so nothing needs
 * clearing); calls that overlap on the GPU (different streams, or graph
 * replays in flight together) race on it and must be serialised. */
int softmax_xent_noalloc_max_batch(void);
mlp_status softmax_xent_fwd_bwd_noalloc(const float* logits, int ld_logits,
                                        const int32_t* labels, int batch, int classes,
                                        float* loss_out, void* dlogits, int dlogits_dtype,
                                        int ld_dlogits, int32_t* argmax_out, void* stream);

/* ---------------------------------------------------------------- update ---
 * Momentum SGD over one flat buffer ([cap] "Read the worked reference"):
 *   v <- momentum * v - lr * g;  w <- w + v.
 * w, g, v fp32[n]; w_bf16 (nullable) bf16[n] receives bf16(w) at the same
 * index.  128-bit vectorised over the 16-byte-aligned body, scalar tail. */
mlp_status sgd_momentum_step(float* w, const float* g, float* v, void* w_bf16, size_t n,
                             float lr, float momentum, void* stream);

/* ---------------------------------------------------------------- GEMM -----
 * C[M][N] = epilogue( sum_k A(m,k) B(k,n) ).
 *   a_trans = 0: A stored [M][lda];  a_trans = 1: A stored [K][lda] (A = S^T).
 *   b_trans = 0: B stored [K][ldb];  b_trans = 1: B stored [N][ldb] (B = S^T).
 * ([cap] "Work through the backward pass": the weight and input gradients are
 * multiplies with one transposed input; no transpose copy is made.)
 * in_dtype F32 runs the fp32 SIMT kernel; BF16 and F16 run the tcgen05 kernel
 * (bf16 or fp16 operands from TMA, fp32 accumulation in tensor memory).
 * Epilogue, in fp32, in this order ([cap] "Read the worked reference"; [vk]):
 *   + bias[n] (nullable, fp32);  act (NONE or RELU);
 *   mask (nullable, dtype = in_dtype, [M][ldm]): keep where mask > 0, else 0;
 *   store as c_dtype into C [M][ldc]: F32, or the 16-bit type of the operands
 *   (BF16 for in_dtype F32 or BF16, F16 for in_dtype F16).
 * K = 0 gives the epilogue of a zero sum. */
mlp_status mlp_gemm(int M, int N, int K, const void* A, int lda, int a_trans, const void* B,
                    int ldb, int b_trans, int in_dtype, const float* bias, int act,
                    const void* mask, int ldm, void* C, int ldc, int c_dtype, void* stream);

/* Column reduction: out[c] = sum_r X[r][c] in fp32 (bias gradient, [cap]
 * "Check your mapping": one bias per unit, summed over the batch).  X dtype
 * F32, BF16 or F16, [rows][ld].  Fixed-order two-pass reduction (bitwise
 * reproducible); workspace: mlp_colsum_workspace_bytes(rows, cols). */
size_t mlp_colsum_workspace_bytes(int rows, int cols);
mlp_status mlp_colsum(const void* X, int dtype, int rows, int cols, int ld, float* out,
                      void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- attention prep
 * The fused attention preprocessing of [mk] "What Worked" (QK RMSNorm +
 * partial RoPE + q gain after the projection) in the fully fused form that
 * [mk] "What Didn't Work" finds achievable in raw CUDA (RMSNorm -> QKV
 * projection -> QK norm -> RoPE -> gain).  Per token t at position
 * p = t mod seq_len:
 *   r = 1 / sqrt(mean_i x_i^2 + eps);  u = r (x W_qkv)          (RMSNorm, gain 1)
 *   u = [n_q query heads | n_kv key heads | n_kv value heads] of head_dim;
 *   query and key heads: u_h <- u_h / sqrt(mean_j u_hj^2 + eps)  (QK norm, gain 1)
 *     then for i < rope_dims / 2, with a = p * rope_theta^(-2i / rope_dims):
 *     (u_i, u_{i+R/2}) <- (u_i cos a - u_{i+R/2} sin a, u_{i+R/2} cos a + u_i sin a)
 *     (rotate-half RoPE on the first rope_dims dims of the head);
 *   query heads: u_h <- q_gain[h] u_h;  value heads: unchanged.
 * x bf16 [T][d]; w_qkv bf16 [d][N] with N = (n_q_heads + 2 n_kv_heads) *
 * head_dim; q_gain fp32 [n_q_heads]; qkv_out bf16 [T][N]; rstd_out fp32 [T]
 * receives r (it is also the kernels' scratch).  Two launches: the per-token
 * r, then the tcgen05 projection whose epilogue applies r, the QK norm, RoPE
 * and the gain to each head while it is in registers.
 * Supported: head_dim 64, rope_dims 16, 32 or 64, d a multiple of 8.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED (16-byte base pointers). */
mlp_status mlp_attn_prep_fwd(const void* x, const void* w_qkv, const float* q_gain, int T,
                             int d, int n_q_heads, int n_kv_heads, int head_dim, int rope_dims,
                             int seq_len, float eps, float rope_theta, void* qkv_out,
                             float* rstd_out, void* stream);

/* ---------------------------------------------------------------- block ----
 * Transformer MLP block ([mk] "What Worked"), per token t:
 *   r = 1 / sqrt(mean_i x_i^2 + eps);  n = r x          (RMSNorm, gain 1)
 *   u = n W_gate;  a = f(u), f(u) = (u > 0 ? u : slope u)^2   (LeakyReLU^2)
 *   y = x + a W_down                                    (residual)
 * x, y bf16 [T][d]; W_gate bf16 [d][hidden]; W_down bf16 [hidden][d];
 * rstd_out fp32 [T] (nullable) receives r.  The [T][hidden] intermediate is
 * never written to memory: it lives in tensor memory and shared memory.
 * Supported: d == 512, hidden a multiple of 256, T any size. */
mlp_status mlp_block_fwd(const void* x, const void* w_gate, const void* w_down, int T, int d,
                         int hidden, float eps, float slope, void* y, float* rstd_out,
                         void* stream);

/* Backward of the block given dy = dL/dy (bf16 [T][d]) and the forward's
 * rstd (fp32 [T]):
 *   da = dy W_down^T;  du = da * f'(u);  dW_down = a^T dy;  dW_gate = n^T du;
 *   dn = du W_gate^T;  dx = dy + r (dn - n mean_i(dn_i n_i)).
 * u is recomputed from x and rstd.  dx bf16 [T][d]; dw_gate fp32 [d][hidden];
 * dw_down fp32 [hidden][d] (overwritten).  workspace holds the bf16 a and
 * r*du tensors for the two weight-gradient GEMMs. */
size_t mlp_block_workspace_bytes(int T, int d, int hidden);
mlp_status mlp_block_bwd(const void* x, const float* rstd, const void* w_gate,
                         const void* w_down, const void* dy, int T, int d, int hidden, float eps,
                         float slope, void* dx, float* dw_gate, float* dw_down, void* workspace,
                         size_t ws_bytes, void* stream);

/* Mean-squared loss: loss = mean((y - t)^2) over n elements, dy = 2 (y - t) / n.
 * y, t, dy bf16[n]; loss_out device fp32 scalar; fixed-order reduction. */
size_t mse_workspace_bytes(size_t n);
mlp_status mse_loss_fwd_bwd(const void* y, const void* t, size_t n, float* loss_out, void* dy,
                            void* workspace, size_t ws_bytes, void* stream);

/* One training step of a stack of n_blocks blocks over T tokens with the
 * mean-squared loss on the last output: block forwards (saving each block
 * input and rstd in the workspace), MSE, block backwards in reverse order
 * (the first block's without its input gradient, which the step does not
 * return), then momentum SGD with the bf16 shadow refresh.
 * params, velocity, grads: fp32, per block W_gate [d][hidden] then
 * W_down [hidden][d]; params_bf16: bf16 shadow in the same layout.
 * x0, target: bf16 [T][d].  loss_out: device fp32 scalar. */
size_t mlp_stack_param_count(int n_blocks, int d, int hidden);
size_t mlp_stack_workspace_bytes(int n_blocks, int T, int d, int hidden);
mlp_status mlp_stack_train_step(int n_blocks, int T, int d, int hidden, float eps, float slope,
                                const void* x0, const void* target, float* params,
                                float* velocity, float* grads, void* params_bf16, float lr,
                                float momentum, float* loss_out, void* workspace,
                                size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLP_STEP_H */
