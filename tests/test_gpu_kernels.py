"""Parity of the single kernels (through the C ABI) with the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import mlp_step_gb300 as M
from mlp_step_gb300 import synth
from helpers import values16, bf16_values, to_dev, rel_to_max, assert_elementwise, near_tie_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    M.load()
    yield
    assert M.get_device_status() == M.MLP_OK


# ------------------------------------------------------------------ SGD

@pytest.mark.parametrize("n", [203530, 1001, 3, 4 * 1024 * 1024 + 5])
def test_sgd_matches_oracle(n):
    lr, m = 0.1, 0.9
    w = synth.normal_f32((n,), synth.STREAM_GENERIC)
    g = synth.normal_f32((n,), synth.STREAM_GENERIC + 1)
    v = synth.normal_f32((n,), synth.STREAM_GENERIC + 2, std=0.01)
    wd, gd, vd = to_dev(w), to_dev(g), to_dev(v)
    wb = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    M.sgd_momentum_step(wd, gd, vd, lr, m, w_bf16=wb)
    w_ref, v_ref = oracle.sgd_momentum(w, g, v, lr, m)
    # "Stage 2: backward and update" (case 5): |got - ref| <= 1e-6 + 1e-5 |ref|
    assert_elementwise(wd.cpu().numpy(), w_ref, 1e-5, 1e-6, "w")
    assert_elementwise(vd.cpu().numpy(), v_ref, 1e-5, 1e-6, "v")
    # the shadow is bf16 of the updated fp32 weight, element for element
    assert torch.equal(wb, wd.to(torch.bfloat16))


def test_sgd_two_steps_closed_form():
    n, lr, m = 4099, 0.1, 0.9
    w0 = synth.normal_f32((n,), synth.STREAM_GENERIC)
    g0 = synth.normal_f32((n,), synth.STREAM_GENERIC + 1)
    g1 = synth.normal_f32((n,), synth.STREAM_GENERIC + 2)
    wd, vd = to_dev(w0), torch.zeros(n, device="cuda")
    M.sgd_momentum_step(wd, to_dev(g0), vd, lr, m)
    M.sgd_momentum_step(wd, to_dev(g1), vd, lr, m)
    w0d, g0d, g1d = (a.astype(np.float64) for a in (w0, g0, g1))
    assert_elementwise(wd.cpu().numpy(), w0d - lr * g0d * (1 + m) - lr * g1d, 1e-5, 1e-6, "w2")


# ------------------------------------------------------------------ softmax xent

def _xent_case(B, C, Z, y, dl_dtype):
    ld = (C + 7) // 8 * 8
    Zd = to_dev(Z)
    yd = to_dev(y)
    loss = torch.zeros(1, device="cuda")
    dl = torch.full((B, ld), 7.0, dtype=dl_dtype, device="cuda")
    am = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(M.softmax_xent_workspace_bytes(B, C), 16), dtype=torch.uint8,
                     device="cuda")
    M.softmax_xent_fwd_bwd(Zd, yd, loss, dlogits=dl, argmax_out=am, workspace=ws, classes=C)
    return loss.item(), dl.float().cpu().numpy(), am.cpu().numpy()


@pytest.mark.parametrize("B,C", [(128, 10), (112, 10), (1, 10), (300, 10), (16384, 1000),
                                 (257, 1000)])
def test_xent_matches_oracle(B, C):
    Z = synth.normal_f32((B, C), synth.STREAM_GENERIC, std=3.0)
    y = synth.labels(B, C, seed=17)
    loss, dl, am = _xent_case(B, C, Z, y, torch.float32)
    l_ref, _, dZ_ref, am_ref = oracle.softmax_xent(Z.astype(np.float64), y)
    assert abs(loss - l_ref) <= 2e-6 * max(1.0, abs(l_ref))
    assert_elementwise(dl[:, :C], dZ_ref, 1e-5, 1e-7 / B, "dZ")
    assert np.all(dl[:, C:] == 0.0)  # padding columns written as zero
    ok = ~near_tie_rows(Z)
    assert np.array_equal(am[ok], am_ref[ok])


def test_xent_bf16_dlogits():
    B, C = 128, 10
    Z = synth.normal_f32((B, C), synth.STREAM_GENERIC, std=3.0)
    y = synth.labels(B, C, seed=17)
    _, dl, _ = _xent_case(B, C, Z, y, torch.bfloat16)
    _, _, dZ_ref, _ = oracle.softmax_xent(Z.astype(np.float64), y)
    assert rel_to_max(dl[:, :C], dZ_ref) <= 4e-3


@pytest.mark.parametrize("B,C", [(128, 10), (300, 1000)])
def test_xent_f16_dlogits(B, C):
    Z = synth.normal_f32((B, C), synth.STREAM_GENERIC, std=3.0)
    y = synth.labels(B, C, seed=17)
    _, dl, _ = _xent_case(B, C, Z, y, torch.float16)
    _, _, dZ_ref, _ = oracle.softmax_xent(Z.astype(np.float64), y)
    # fp16: 11 significant bits, subnormal below 2^-14 (dZ carries 1 / B)
    assert_elementwise(dl[:, :C], dZ_ref, 1e-3, 2.0 ** -24, "dZ")


def test_xent_extreme_logits_pm60():
    # "Capstone 5", "Read the worked reference": logits at +/-60 must give
    # finite loss and gradients; closed forms per row (k entries at +60).
    B, C = 200, 10
    Z, k = synth.logits_pm60(B, C)
    y = synth.labels(B, C, seed=5)
    loss, dl, am = _xent_case(B, C, Z, y, torch.float32)
    assert math.isfinite(loss) and np.all(np.isfinite(dl))
    top = Z[np.arange(B), y] > 0
    want = np.where(top, np.log(k), 120.0 + np.log(k)).mean()
    assert abs(loss - want) <= 1e-5 * want
    p = dl[:, :C] * B + (np.arange(C)[None, :] == y[:, None])
    pos = Z > 0
    assert np.allclose(p[pos], np.repeat(1.0 / k, (pos).sum(1)), rtol=1e-5)
    am_ref = np.argmax(Z, 1)  # first +60
    assert np.array_equal(am, am_ref)


@pytest.mark.parametrize("B,C,ld", [(1000, 250, 256), (600, 1001, 1008), (700, 130, 132)])
def test_xent_rows_ragged_classes_in_padded_pitch(B, C, ld):
    """Batches above 256 rows take the row-buffered warp kernel (rows of up to
    256 or 1,024 classes).  Rows of C classes in a wider pitch whose padding
    holds huge logits: the classes past C must not reach the max, the sum or
    dZ (C not a multiple of 4 exercises the masking of the copied padding).
    The call without argmax (plain row max) gives the same loss and dZ bit
    for bit."""
    Z = synth.normal_f32((B, C), synth.STREAM_GENERIC + 7, std=3.0)
    y = synth.labels(B, C, seed=23)
    Zp = np.full((B, ld), 1e30, dtype=np.float32)
    Zp[:, :C] = Z
    Zd, yd = to_dev(Zp), to_dev(y)
    ldd = (C + 7) // 8 * 8
    ws = torch.empty(max(M.softmax_xent_workspace_bytes(B, C), 16), dtype=torch.uint8,
                     device="cuda")
    outs = []
    for with_argmax in (True, False):
        loss = torch.zeros(1, device="cuda")
        dl = torch.full((B, ldd), 7.0, dtype=torch.float32, device="cuda")
        am = torch.empty(B, dtype=torch.int32, device="cuda") if with_argmax else None
        M.softmax_xent_fwd_bwd(Zd, yd, loss, dlogits=dl, argmax_out=am, workspace=ws, classes=C)
        outs.append((loss.item(), dl.cpu().numpy(), am.cpu().numpy() if with_argmax else None))
    l_ref, _, dZ_ref, am_ref = oracle.softmax_xent(Z.astype(np.float64), y)
    loss, dl, am = outs[0]
    assert abs(loss - l_ref) <= 2e-6 * max(1.0, abs(l_ref))
    assert_elementwise(dl[:, :C], dZ_ref, 1e-5, 1e-7 / B, "dZ")
    assert np.all(dl[:, C:] == 0.0)
    ok = ~near_tie_rows(Z)
    assert np.array_equal(am[ok], am_ref[ok])
    assert outs[1][0] == loss and np.array_equal(outs[1][1], dl)


# ------------------------------------------------------------------ column sums

@pytest.mark.parametrize("rows,cols,dtype", [(128, 10, torch.float32), (128, 256, torch.bfloat16),
                                             (16384, 1000, torch.bfloat16), (3, 5, torch.float32),
                                             (1, 64, torch.bfloat16), (5000, 333, torch.float32),
                                             (16384, 1000, torch.float16), (7, 13, torch.float16)])
def test_colsum_matches_oracle(rows, cols, dtype):
    X = synth.normal_f32((rows, cols), synth.STREAM_GENERIC)
    Xd = to_dev(X, dtype)
    out = torch.empty(cols, device="cuda")
    ws = torch.empty(max(M.mlp_colsum_workspace_bytes(rows, cols), 16), dtype=torch.uint8,
                     device="cuda")
    M.mlp_colsum(Xd, out, workspace=ws)
    ref = oracle.colsum(Xd.float().cpu().numpy())
    # fp32 accumulation of `rows` terms of magnitude ~1
    assert_elementwise(out.cpu().numpy(), ref, 1e-5, 1e-6 * math.sqrt(rows), "colsum")


# ------------------------------------------------------------------ GEMM (fp32 SIMT)

def _operands(M_, N, K, a_t, b_t, seed=0):
    A = synth.normal_f32((K, M_) if a_t else (M_, K), synth.STREAM_GENERIC + seed)
    B = synth.normal_f32((N, K) if b_t else (K, N), synth.STREAM_GENERIC + seed + 1)
    return A, B


@pytest.mark.parametrize("a_t,b_t", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("shape", [(128, 256, 784), (67, 33, 129), (1, 10, 256), (784, 256, 128)])
def test_gemm_fp32_matches_oracle(shape, a_t, b_t):
    M_, N, K = shape
    A, B = _operands(M_, N, K, a_t, b_t)
    bias = synth.normal_f32((N,), synth.STREAM_GENERIC + 5)
    C = torch.empty(M_, N, device="cuda")
    M.mlp_gemm(to_dev(A), to_dev(B), C, M_, N, K, a_trans=a_t, b_trans=b_t, bias=to_dev(bias),
               act=M.MLP_ACT_RELU)
    ref = np.maximum(oracle.matmul(A, B, a_t=bool(a_t), b_t=bool(b_t)) + bias, 0.0)
    assert_elementwise(C.cpu().numpy(), ref, 1e-5, 1e-5 * math.sqrt(K), "C")


# ------------------------------------------------------------------ GEMM (bf16 tcgen05)

def _tc_case(M_, N, K, a_t, b_t, bias=False, act=M.MLP_ACT_NONE, mask=False, out_bf16=False,
             seed=0, h16=torch.bfloat16):
    """One tensor-core GEMM with 16-bit operands of type h16 (bf16 or fp16);
    out_bf16 selects a 16-bit output of the same type."""
    A, B = _operands(M_, N, K, a_t, b_t, seed)
    Ad, Bd = to_dev(A, h16), to_dev(B, h16)
    bvec = synth.normal_f32((N,), synth.STREAM_GENERIC + 5) if bias else None
    mk = synth.normal_f32((M_, N), synth.STREAM_GENERIC + 6) if mask else None
    C = torch.full((M_, N), float("nan"), dtype=h16 if out_bf16 else torch.float32,
                   device="cuda")
    M.mlp_gemm(Ad, Bd, C, M_, N, K, a_trans=a_t, b_trans=b_t,
               bias=to_dev(bvec) if bias else None, act=act,
               mask=to_dev(mk, h16) if mask else None)
    ref = oracle.matmul(values16(A, h16), values16(B, h16), a_t=bool(a_t), b_t=bool(b_t))
    if bias:
        ref = ref + bvec
    if act == M.MLP_ACT_RELU:
        ref = np.maximum(ref, 0.0)
    if mask:
        ref = np.where(values16(mk, h16) > 0, ref, 0.0)
    return C.float().cpu().numpy(), ref


@pytest.mark.parametrize("a_t,b_t", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("shape", [(128, 256, 784), (300, 200, 136), (129, 65, 64), (1, 16, 8),
                                   (256, 10, 128), (128, 256, 10), (2560, 1024, 192),
                                   (640, 768, 320),
                                   # CTA-pair 256 x 256 tiles: whole tiles, ragged M / N / K
                                   # (the last pair tile's odd CTA entirely past M), and
                                   # an output row pitch that rules out TMA stores
                                   (2304, 1536, 200), (2100, 1800, 72), (2100, 1803, 72)])
def test_gemm_bf16_tc_matches_oracle(shape, a_t, b_t):
    M_, N, K = shape
    if (not a_t and K % 8) or (a_t and M_ % 8) or (not b_t and N % 8) or (b_t and K % 8):
        pytest.skip("bf16 rows must be 16-byte aligned for TMA")
    got, ref = _tc_case(M_, N, K, a_t, b_t)
    assert np.all(np.isfinite(got)), "unwritten outputs"
    assert rel_to_max(got, ref) <= 1e-5, rel_to_max(got, ref)


@pytest.mark.parametrize("bias,act,mask,out_bf16", [(True, M.MLP_ACT_RELU, False, True),
                                                    (False, M.MLP_ACT_NONE, True, True),
                                                    (True, M.MLP_ACT_NONE, False, False)])
def test_gemm_bf16_tc_epilogues(bias, act, mask, out_bf16):
    got, ref = _tc_case(333, 520, 200, 0, 0, bias=bias, act=act, mask=mask, out_bf16=out_bf16)
    tol = 8e-3 if out_bf16 else 1e-5
    assert rel_to_max(got, ref) <= tol
    if act == M.MLP_ACT_RELU:
        assert np.all(got >= 0)
    if mask:
        mk = synth.normal_f32((333, 520), synth.STREAM_GENERIC + 6)
        assert np.all(got[bf16_values(mk) <= 0] == 0)


@pytest.mark.parametrize("out_bf16", [False, True])
@pytest.mark.parametrize("shape", [(1100, 1000, 136), (1029, 1032, 64), (2100, 1800, 72)])
def test_gemm_bf16_tc_large_ragged_outputs(shape, out_bf16):
    # outputs of a million elements or more leave through TMA bulk stores;
    # the ragged last tiles must be clipped exactly
    M_, N, K = shape
    got, ref = _tc_case(M_, N, K, 0, 0, bias=True, act=M.MLP_ACT_RELU, out_bf16=out_bf16)
    assert np.all(np.isfinite(got)), "unwritten outputs"
    assert rel_to_max(got, ref) <= (8e-3 if out_bf16 else 1e-5)


@pytest.mark.parametrize("a_t,b_t", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("shape", [(128, 256, 784), (300, 200, 136), (1, 16, 8), (256, 10, 128),
                                   (2304, 1536, 200), (2100, 1803, 72)])
def test_gemm_f16_tc_matches_oracle(shape, a_t, b_t):
    """fp16 operands ("The Debugging Lesson Was Numerical": FP16 in, FP32
    accumulate) through the same single-CTA and CTA-pair kernels."""
    M_, N, K = shape
    if (not a_t and K % 8) or (a_t and M_ % 8) or (not b_t and N % 8) or (b_t and K % 8):
        pytest.skip("fp16 rows must be 16-byte aligned for TMA")
    got, ref = _tc_case(M_, N, K, a_t, b_t, h16=torch.float16)
    assert np.all(np.isfinite(got)), "unwritten outputs"
    assert rel_to_max(got, ref) <= 1e-5, rel_to_max(got, ref)


@pytest.mark.parametrize("bias,act,mask,out16", [(True, M.MLP_ACT_RELU, False, True),
                                                 (False, M.MLP_ACT_NONE, True, True),
                                                 (True, M.MLP_ACT_NONE, False, False)])
def test_gemm_f16_tc_epilogues(bias, act, mask, out16):
    got, ref = _tc_case(333, 520, 200, 0, 0, bias=bias, act=act, mask=mask, out_bf16=out16,
                        h16=torch.float16)
    # fp16 output: 11 significant bits
    assert rel_to_max(got, ref) <= (1e-3 if out16 else 1e-5)
    if mask:
        mk = synth.normal_f32((333, 520), synth.STREAM_GENERIC + 6)
        assert np.all(got[values16(mk, torch.float16) <= 0] == 0)
    # large outputs leave through TMA bulk stores in the fp16 format
    got, ref = _tc_case(2100, 1800, 72, 0, 0, bias=True, act=M.MLP_ACT_RELU, out_bf16=out16,
                        h16=torch.float16)
    assert rel_to_max(got, ref) <= (1e-3 if out16 else 1e-5)


def test_gemm_bf16_tc_k_zero_gives_bias():
    N = 24
    bias = synth.normal_f32((N,), synth.STREAM_GENERIC + 5)
    C = torch.empty(5, N, device="cuda")
    A = torch.zeros(5, 8, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(8, N, dtype=torch.bfloat16, device="cuda")
    M.mlp_gemm(A, B, C, 5, N, 0, bias=to_dev(bias))
    assert np.array_equal(C.cpu().numpy(), np.tile(bias, (5, 1)))


@pytest.mark.parametrize("h16", [torch.bfloat16, torch.float16])
def test_gemm_16bit_k_zero_writes_bias_in_the_operand_format(h16):
    """K = 0 with a 16-bit output: the epilogue of a zero sum, stored in the
    operands' 16-bit format (bf16 or fp16)."""
    N = 24
    bias = synth.normal_f32((N,), synth.STREAM_GENERIC + 5)
    C = torch.full((5, N), float("nan"), dtype=h16, device="cuda")
    A = torch.zeros(5, 8, dtype=h16, device="cuda")
    B = torch.zeros(8, N, dtype=h16, device="cuda")
    M.mlp_gemm(A, B, C, 5, N, 0, bias=to_dev(bias), act=M.MLP_ACT_RELU)
    want = torch.from_numpy(np.tile(np.maximum(bias, 0.0), (5, 1))).to(h16)
    assert torch.equal(C.cpu(), want)


def test_gemm_bf16_tc_deterministic():
    A, B = _operands(1000, 1000, 1000, 0, 0)
    Ad, Bd = to_dev(A, torch.bfloat16), to_dev(B, torch.bfloat16)
    C1 = torch.empty(1000, 1000, device="cuda")
    C2 = torch.empty(1000, 1000, device="cuda")
    M.mlp_gemm(Ad, Bd, C1, 1000, 1000, 1000)
    M.mlp_gemm(Ad, Bd, C2, 1000, 1000, 1000)
    assert torch.equal(C1, C2)


# ------------------------------------------------------------------ bounded wait

def test_bounded_wait_times_out_cleanly():
    M.selftest_wait_timeout(20_000_000)  # 20 ms
    assert M.get_device_status() == M.MLP_ERR_DEVICE_TIMEOUT
    assert M.get_device_status() == M.MLP_OK  # cleared, context still usable
    x = torch.ones(4, device="cuda")
    assert x.sum().item() == 4.0


# ------------------------------------------------------------------ linear order

@pytest.fixture
def linear_order():
    M.set_reduction_order(M.MLP_ORDER_LINEAR)
    yield
    M.set_reduction_order(M.MLP_ORDER_FAST)


@pytest.mark.parametrize("a_t,b_t", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("shape", [(128, 256, 784), (67, 33, 129), (785, 256, 128), (1, 10, 256)])
def test_gemm_fp32_linear_order_is_bit_exact(shape, a_t, b_t, linear_order):
    """MLP_ORDER_LINEAR ("HIP + Vulkan backends -- Phase 3", "Phase-3 bug
    hunt": linear-order sums for bit parity): each output is one fused
    multiply-add chain over ascending k, + bias, ReLU, mask -- the oracle's
    fp32 chain to the bit (these shapes split K in the default mode)."""
    M_, N, K = shape
    A, B = _operands(M_, N, K, a_t, b_t)
    bias = synth.normal_f32((N,), synth.STREAM_GENERIC + 5)
    mk = synth.normal_f32((M_, N), synth.STREAM_GENERIC + 6)
    C = torch.full((M_, N), float("nan"), device="cuda")
    M.mlp_gemm(to_dev(A), to_dev(B), C, M_, N, K, a_trans=a_t, b_trans=b_t, bias=to_dev(bias),
               act=M.MLP_ACT_RELU, mask=to_dev(mk))
    want = oracle.matmul_f32_linear(A, B, a_t=a_t, b_t=b_t, bias=bias, act=1, mask=mk)
    got = C.cpu().numpy()
    assert np.array_equal(got, want), np.abs(got - want).max()


@pytest.mark.parametrize("rows,cols,dtype", [(16384, 1000, torch.float32), (5000, 333, torch.float32),
                                             (128, 256, torch.bfloat16), (7, 13, torch.float16)])
def test_colsum_linear_order_is_bit_exact(rows, cols, dtype, linear_order):
    X = synth.normal_f32((rows, cols), synth.STREAM_GENERIC)
    Xd = to_dev(X, dtype)
    out = torch.empty(cols, device="cuda")
    ws = torch.empty(max(M.mlp_colsum_workspace_bytes(rows, cols), 16), dtype=torch.uint8,
                     device="cuda")
    M.mlp_colsum(Xd, out, workspace=ws)
    want = oracle.colsum_f32_linear(Xd.float().cpu().numpy())
    assert np.array_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("B,C", [(100, 10), (200, 1000), (3000, 1000)])
@pytest.mark.parametrize("bad", [float("inf"), float("nan")])
def test_xent_nonfinite_logits_report_numeric(B, C, bad):
    """Logits holding an infinity or a NaN give a non-finite loss; every path
    of the loss kernel (one row per thread, one block, per-block partials)
    records it for mlp_get_device_status as MLP_ERR_NUMERIC."""
    Z = torch.from_numpy(synth.normal_f32((B, C), synth.STREAM_GENERIC + 9)).cuda()
    Z[B // 2, 1] = bad
    y = torch.from_numpy(synth.labels(B, C)).cuda()
    loss = torch.zeros(4, device="cuda")
    ws = torch.empty(max(M.softmax_xent_workspace_bytes(B, C), 16), dtype=torch.uint8,
                     device="cuda")
    M.softmax_xent_fwd_bwd(Z, y, loss, workspace=ws)
    assert M.get_device_status() == M.MLP_ERR_NUMERIC
    assert M.get_device_status() == M.MLP_OK
    Z[B // 2, 1] = 0.0
    M.softmax_xent_fwd_bwd(Z, y, loss, workspace=ws)
    assert M.get_device_status() == M.MLP_OK
    assert np.isfinite(loss[0].item())


def test_mse_nonfinite_output_reports_numeric():
    n = 512 * 64
    yv = torch.from_numpy(synth.normal_f32((n,), synth.STREAM_BLOCK_X)).to(torch.bfloat16).cuda()
    t = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    yv[77] = float("nan")
    loss = torch.zeros(4, device="cuda")
    dy = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(M.mse_workspace_bytes(n), dtype=torch.uint8, device="cuda")
    M.mse_loss_fwd_bwd(yv, t, loss, dy, ws)
    assert M.get_device_status() == M.MLP_ERR_NUMERIC
    assert M.get_device_status() == M.MLP_OK
