"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test ties one oracle function to something the pages print, a closed form,
an invariant, a central finite difference, or a library routine in a special
case.  A plausible slip in the oracle (a dropped bias, a wrong sign, a
transposed operand, a missing 1/B, a wrong mask) fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
from mlp_step_gb300 import synth

DIMS = [784, 256, 10]


# ------------------------------------------------------------ printed facts

def test_param_count_printed(golden):
    assert oracle.param_count(DIMS) == golden["param_count_784_256_10"]["value"]
    # the wide MLP and the block stack, by the same definition
    assert oracle.param_count([1024, 8192, 8192, 1000]) == 83_706_856


def test_bf16_rounding_matches_library():
    import torch
    x = synth.normal(7, synth.STREAM_GENERIC, 20000) * np.exp(synth.normal(7, synth.STREAM_GENERIC + 1, 20000))
    x32 = x.astype(np.float32)
    want = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in x32])
    assert np.array_equal(got, want)
    # ties to even at 1 + 2^-8 and 1 + 3*2^-8
    assert oracle.round_bf16(1 + 2 ** -8) == 1.0
    assert oracle.round_bf16(1 + 3 * 2 ** -8) == 1 + 2 ** -6


def test_f16_rounding_matches_library_and_binary16_edges():
    # numpy converts float64 to IEEE binary16 in one correctly rounded step
    mag = np.exp(4.0 * synth.normal(9, synth.STREAM_GENERIC + 1, 20000))
    x = synth.normal(9, synth.STREAM_GENERIC, 20000) * mag
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).astype(np.float64)
    got = np.array([oracle.round_f16(float(v)) for v in x])
    assert np.array_equal(got, want)
    assert np.isinf(got).any() and (np.abs(got[got != 0]) < 2.0 ** -14).any()  # both ends hit
    # values fixed by the binary16 format: largest finite 65504 = (2 - 2^-10) 2^15;
    # halfway to the next step (65520) rounds to infinity; subnormal step 2^-24
    assert oracle.round_f16(65504.0) == 65504.0
    assert oracle.round_f16(65519.99) == 65504.0
    assert oracle.round_f16(65520.0) == math.inf
    assert oracle.round_f16(-65520.0) == -math.inf
    assert oracle.round_f16(2.0 ** -24) == 2.0 ** -24
    assert oracle.round_f16(2.0 ** -25) == 0.0               # tie between 0 and 2^-24: even
    assert oracle.round_f16(3 * 2.0 ** -25) == 2.0 ** -23    # tie between 2^-24 and 2^-23
    assert oracle.round_f16(1 + 2.0 ** -11) == 1.0            # ties to even above 1
    assert oracle.round_f16(1 + 3 * 2.0 ** -11) == 1 + 2.0 ** -9
    assert oracle.round_f16(1.0 / 3.0) == 1365.0 / 4096.0     # 0x3555


def test_rounding_points_modes_round_where_the_formats_differ():
    """With identity weights the logits are the inputs.  1 + 2^-9 has 10
    significant bits: binary16 holds it (fp16 points agree with exact mode),
    bf16 does not (8 bits: it becomes 1).  1 + 2^-12 fits neither."""
    dims = [2, 2, 2]
    params = np.zeros(oracle.param_count(dims))
    params[0:4] = [1, 0, 0, 1]        # W1 = I
    params[6:10] = [1, 0, 0, 1]       # W2 = I
    X = np.array([[1 + 2.0 ** -9, 1 + 2.0 ** -12]])
    _, z_exact = oracle.mlp_forward(dims, params, X)
    _, z_f16 = oracle.mlp_forward(dims, params, X, points="f16")
    _, z_bf16 = oracle.mlp_forward(dims, params, X, points="bf16")
    assert z_exact[0].tolist() == [1 + 2.0 ** -9, 1 + 2.0 ** -12]
    assert z_f16[0].tolist() == [1 + 2.0 ** -9, 1.0]
    assert z_bf16[0].tolist() == [1.0, 1.0]
    assert oracle.mlp_forward(dims, params, X, bf16_points=True)[1].tolist() == z_bf16.tolist()


# ------------------------------------------------------------ GEMM

def test_linear_f32_matmul_is_one_fused_chain_per_output():
    """The linear-order fp32 GEMM: one fused multiply-add chain over ascending
    k per output.  With a = [1, 1 + 2^-12] and b = [-(1 + 2^-11), 1 + 2^-12]
    the exact dot product is 2^-24; the chain's second step fma((1 + 2^-12)^2,
    -(1 + 2^-11)) keeps it, while rounding the product first (a tie at half an
    ulp of 1, to even) would give 0."""
    a = np.array([[1.0, 1 + 2.0 ** -12]], dtype=np.float32)
    b = np.array([[-(1 + 2.0 ** -11)], [1 + 2.0 ** -12]], dtype=np.float32)
    assert oracle.matmul_f32_linear(a, b)[0, 0] == np.float32(2.0 ** -24)
    # integer operands: every partial sum is an integer below 2^24, exact in
    # fp32, so the chain equals the fp64 product for every operand layout
    M_, N, K = 5, 7, 9
    A = np.floor(synth.uniform01(3, synth.STREAM_GENERIC, M_ * K) * 19 - 9).reshape(M_, K)
    B = np.floor(synth.uniform01(3, synth.STREAM_GENERIC + 1, K * N) * 19 - 9).reshape(K, N)
    bias = np.floor(synth.uniform01(3, synth.STREAM_GENERIC + 2, N) * 9 - 4)
    mask = np.floor(synth.uniform01(3, synth.STREAM_GENERIC + 3, M_ * N) * 3 - 1).reshape(M_, N)
    want = np.where(mask > 0, np.maximum(A @ B + bias, 0.0), 0.0)
    for a_t in (0, 1):
        for b_t in (0, 1):
            got = oracle.matmul_f32_linear(A.T if a_t else A, B.T if b_t else B, a_t=a_t,
                                           b_t=b_t, bias=bias, act=1, mask=mask)
            assert np.array_equal(got, want), (a_t, b_t)


def test_linear_f32_colsum_adds_rows_in_ascending_order():
    """1 + 1e8 rounds back to 1e8 in fp32 (ulp 8), so adding [1, 1e8, -1e8]
    from the top gives 0 although the exact sum is 1 (from the bottom: 1)."""
    X = np.array([[1.0, -3.0], [1e8, 2.0], [-1e8, 5.0]], dtype=np.float32)
    assert oracle.colsum_f32_linear(X).tolist() == [0.0, 4.0]
    Xi = np.floor(synth.uniform01(4, synth.STREAM_GENERIC, 300 * 7) * 201 - 100).reshape(300, 7)
    assert np.array_equal(oracle.colsum_f32_linear(Xi), Xi.sum(0))


@pytest.mark.parametrize("a_t,b_t", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_matmul_matches_library(a_t, b_t):
    M, N, K = 7, 5, 11
    A = synth.normal(1, synth.STREAM_GENERIC, M * K).reshape((K, M) if a_t else (M, K))
    B = synth.normal(1, synth.STREAM_GENERIC + 1, K * N).reshape((N, K) if b_t else (K, N))
    want = (A.T if a_t else A) @ (B.T if b_t else B)
    got = oracle.matmul(A, B, a_t=bool(a_t), b_t=bool(b_t))
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13)
    ii = np.array([0, 6, 3]); jj = np.array([4, 0, 2])
    ent = oracle.matmul_entries(A, B, ii, jj, a_t=bool(a_t), b_t=bool(b_t))
    want32 = (A.astype(np.float32).astype(np.float64).T if a_t else A.astype(np.float32).astype(np.float64)) @ \
             (B.astype(np.float32).astype(np.float64).T if b_t else B.astype(np.float32).astype(np.float64))
    assert np.allclose(ent, want32[ii, jj], rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("a_t,b_t", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_matmul_sums_each_entry_in_ascending_k(a_t, b_t):
    """Every entry is the K products added one at a time in ascending k from
    0.0, as a plain triple loop does, at shapes that cross the row and column
    blocks the oracle's loops visit (bit for bit)."""
    for M, N, K in ((9, 257, 5), (17, 3, 13), (1, 513, 2)):
        A = synth.normal(2, synth.STREAM_GENERIC, M * K).reshape((K, M) if a_t else (M, K))
        B = synth.normal(2, synth.STREAM_GENERIC + 1, K * N).reshape((N, K) if b_t else (K, N))
        Am = A.T if a_t else A
        Bm = B.T if b_t else B
        want = np.zeros((M, N))
        for m in range(M):
            for n in range(N):
                acc = 0.0
                for k in range(K):
                    acc = acc + float(Am[m, k]) * float(Bm[k, n])
                want[m, n] = acc
        got = oracle.matmul(A, B, a_t=bool(a_t), b_t=bool(b_t))
        assert np.array_equal(got, want), (M, N, K)


def test_colsum_matches_library_and_bias_gradient():
    X = synth.normal(3, synth.STREAM_GENERIC, 37 * 13).reshape(37, 13).astype(np.float32)
    got = oracle.colsum(X)
    assert np.allclose(got, X.astype(np.float64).sum(0), rtol=1e-14, atol=1e-14)
    # it is the bias gradient of the backward pass: db = sum_rows dY
    dims = [5, 4, 13]
    p = synth.mlp_flat_params(dims, seed=2).astype(np.float64)
    X0 = synth.normal(3, synth.STREAM_GENERIC + 1, 37 * 5).reshape(37, 5)
    hs, _ = oracle.mlp_forward(dims, p, X0)
    g = oracle.mlp_backward(dims, p, X0, hs, X.astype(np.float64))
    assert np.allclose(g[-13:], got, rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------ forward

def test_forward_all_positive_reduces_to_affine_maps():
    # With positive inputs, weights and biases ReLU is the identity, so the
    # network is the composition of two affine maps (a library matmul chain).
    dims = [6, 5, 3]
    rng = np.random.default_rng(0)
    W1 = rng.uniform(0.1, 1, (6, 5)); b1 = rng.uniform(0.1, 1, 5)
    W2 = rng.uniform(-1, 1, (5, 3)); b2 = rng.uniform(-1, 1, 3)
    X = rng.uniform(0.1, 1, (4, 6))
    p = np.concatenate([W1.ravel(), b1, W2.ravel(), b2])
    hs, Z = oracle.mlp_forward(dims, p, X)
    assert np.allclose(hs[0], X @ W1 + b1, rtol=1e-13)
    assert np.allclose(Z, (X @ W1 + b1) @ W2 + b2, rtol=1e-13)


def test_forward_relu_zeroes_negative_units():
    dims = [3, 4, 2]
    X = np.ones((2, 3))
    W1 = np.zeros((3, 4)); b1 = np.array([1.0, -1.0, 2.0, -3.0])
    W2 = np.ones((4, 2)); b2 = np.zeros(2)
    p = np.concatenate([W1.ravel(), b1, W2.ravel(), b2])
    hs, Z = oracle.mlp_forward(dims, p, X)
    assert np.array_equal(hs[0], np.tile([1.0, 0.0, 2.0, 0.0], (2, 1)))
    assert np.array_equal(Z, np.full((2, 2), 3.0))


def test_forward_rows_agrees_with_batch_forward():
    dims = [20, 16, 5]
    p = synth.mlp_flat_params(dims, seed=3)
    X = synth.images_u8(9, 20, seed=3).astype(np.float32) / np.float32(255)
    _, Z = oracle.mlp_forward(dims, p, X)
    rows = np.array([8, 0, 4])
    Zr = oracle.mlp_forward_rows(dims, p, X, rows)
    assert np.allclose(Zr, Z[rows], rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------ loss

def test_zero_weights_loss_is_ln10():
    B = 128
    p = np.zeros(oracle.param_count(DIMS))
    X = synth.images_u8(B).astype(np.float64) / 255.0
    y = synth.labels(B, 10)
    hs, Z = oracle.mlp_forward(DIMS, p, X)
    loss, rl, dZ, am = oracle.softmax_xent(Z, y)
    assert abs(loss - math.log(10.0)) < 1e-13
    onehot = np.eye(10)[y]
    assert np.allclose(dZ, (0.1 - onehot) / B, rtol=0, atol=1e-18)
    assert np.array_equal(am, np.zeros(B, dtype=np.int32))  # lowest index among ties
    g = oracle.mlp_backward(DIMS, p, X, hs, dZ)
    nW1 = 784 * 256
    assert np.all(g[:nW1 + 256] == 0.0)            # dH = 0 -> dW1 = 0, db1 = 0
    assert np.all(g[nW1 + 256:nW1 + 256 + 2560] == 0.0)  # H = 0 -> dW2 = 0
    assert np.allclose(g[-10:], ((0.1 - onehot) / B).sum(0), atol=1e-17)


def test_extreme_logits_closed_form(golden):
    mag = golden["extreme_logit_magnitude"]["value"]
    B, C = 64, 10
    Z, k = synth.logits_pm60(B, C)
    assert set(np.unique(Z)) == {mag, -mag}
    y = synth.labels(B, C, seed=11)
    loss, rl, dZ, am = oracle.softmax_xent(Z.astype(np.float64), y)
    for b in range(B):
        on_top = Z[b, y[b]] > 0
        want = math.log(k[b]) if on_top else 2 * mag + math.log(k[b])
        assert abs(rl[b] - want) <= 1e-12 * max(1.0, want)
        p_plus = 1.0 / (k[b] + (C - k[b]) * math.exp(-2 * mag))
        p = dZ[b] * B + (np.arange(C) == y[b])
        top = Z[b] > 0
        other = np.arange(C) != y[b]   # p of the label column loses its digits to the -1
        assert np.allclose(p[top], p_plus, rtol=1e-12)
        assert np.allclose(p[~top & other], math.exp(-2 * mag) * p_plus, rtol=1e-9, atol=0)
    assert np.all(np.isfinite(rl)) and np.all(np.isfinite(dZ))
    assert abs(loss - rl.mean()) < 1e-12


def test_softmax_rows_sum_to_one():
    B, C = 50, 1000
    Z = synth.normal(5, synth.STREAM_GENERIC, B * C).reshape(B, C) * 4
    y = synth.labels(B, C, seed=5)
    _, _, dZ, am = oracle.softmax_xent(Z, y)
    assert np.allclose(dZ.sum(1), 0.0, atol=1e-13 / B)
    assert np.array_equal(am, np.argmax(Z, 1))  # library argmax (first maximum)


# ------------------------------------------------------------ backward: FD

def _loss(dims, p, X, y):
    _, Z = oracle.mlp_forward(dims, p, X)
    return oracle.softmax_xent(Z, y)[0]


def _masks(dims, p, X):
    hs, _ = oracle.mlp_forward(dims, p, X)
    return [h > 0 for h in hs]


def _fd_check(dims, p, X, y, coords, h=1e-6):
    hs, Z = oracle.mlp_forward(dims, p, X)
    _, _, dZ, _ = oracle.softmax_xent(Z, y)
    g = oracle.mlp_backward(dims, p, X, hs, dZ)
    checked = 0
    for i in coords:
        pp = p.copy(); pp[i] += h
        pm = p.copy(); pm[i] -= h
        mp, mm = _masks(dims, pp, X), _masks(dims, pm, X)
        if any(not np.array_equal(a, b) for a, b in zip(mp, mm)):
            continue  # the perturbation crosses a ReLU kink
        fd = (_loss(dims, pp, X, y) - _loss(dims, pm, X, y)) / (2 * h)
        assert abs(g[i] - fd) <= 1e-6 + 1e-5 * abs(fd), (i, g[i], fd)
        checked += 1
    return checked


def test_grad_fd_tiny_all_coordinates():
    dims = [5, 4, 3]
    p = synth.mlp_flat_params(dims, seed=9).astype(np.float64)
    p[20:24] = [0.3, -0.2, 0.1, 0.05]  # nonzero b1 so that b1 is exercised
    X = synth.normal(9, synth.STREAM_GENERIC, 15).reshape(3, 5)
    y = np.array([0, 2, 1], dtype=np.int32)
    n = _fd_check(dims, p, X, y, range(p.size))
    assert n >= p.size - 4


def test_grad_fd_seeded_coordinates_784(golden):
    n_coords = golden["grad_check_coordinates"]["value"]
    B = 16
    p = synth.mlp_flat_params(DIMS).astype(np.float64)
    p[784 * 256:784 * 256 + 256] = synth.normal(2, synth.STREAM_GENERIC, 256) * 0.1
    X = synth.images_u8(B).astype(np.float64) / 255.0
    y = synth.labels(B, 10)
    coords = synth.randint(4, synth.STREAM_GENERIC, n_coords, p.size)
    n = _fd_check(DIMS, p, X, y, coords)
    assert n >= 0.9 * n_coords


def test_grad_input_fd():
    dims = [5, 4, 3]
    p = synth.mlp_flat_params(dims, seed=9).astype(np.float64)
    X = synth.normal(9, synth.STREAM_GENERIC, 15).reshape(3, 5)
    y = np.array([0, 2, 1], dtype=np.int32)
    hs, Z = oracle.mlp_forward(dims, p, X)
    _, _, dZ, _ = oracle.softmax_xent(Z, y)
    _, dX = oracle.mlp_backward(dims, p, X, hs, dZ, want_dx=True)
    h = 1e-6
    for idx in np.ndindex(X.shape):
        Xp = X.copy(); Xp[idx] += h
        Xm = X.copy(); Xm[idx] -= h
        fd = (_loss(dims, p, Xp, y) - _loss(dims, p, Xm, y)) / (2 * h)
        assert abs(dX[idx] - fd) <= 1e-6 + 1e-5 * abs(fd)


def test_relu_mask_dead_unit_has_zero_gradient():
    B = 32
    p = synth.mlp_flat_params(DIMS).astype(np.float64)
    dead = [3, 100, 255]
    p[784 * 256 + np.array(dead)] = -1e6   # b1 so large that H[:, j] = 0 for all rows
    X = synth.images_u8(B).astype(np.float64) / 255.0
    y = synth.labels(B, 10)
    hs, Z = oracle.mlp_forward(DIMS, p, X)
    assert np.all(hs[0][:, dead] == 0.0)
    _, _, dZ, _ = oracle.softmax_xent(Z, y)
    g = oracle.mlp_backward(DIMS, p, X, hs, dZ)
    W1g = g[:784 * 256].reshape(784, 256)
    assert np.all(W1g[:, dead] == 0.0)
    assert np.all(g[784 * 256 + np.array(dead)] == 0.0)
    # live units do receive gradient
    assert np.count_nonzero(W1g[:, 0]) > 0


# ------------------------------------------------------------ SGD

def test_sgd_closed_forms(golden):
    lr, m = golden["recipe"]["lr"], golden["recipe"]["momentum"]
    n = 1001
    w0 = synth.normal(1, synth.STREAM_GENERIC, n)
    g0 = synth.normal(1, synth.STREAM_GENERIC + 1, n)
    g1 = synth.normal(1, synth.STREAM_GENERIC + 2, n)
    w1, v1 = oracle.sgd_momentum(w0, g0, np.zeros(n), lr, m)
    assert np.allclose(w1, w0 - lr * g0, rtol=1e-15, atol=1e-15)
    assert np.allclose(v1, -lr * g0, rtol=1e-15, atol=0)
    w2, _ = oracle.sgd_momentum(w1, g1, v1, lr, m)
    assert np.allclose(w2, w0 - lr * g0 * (1 + m) - lr * g1, rtol=1e-13, atol=1e-15)


def test_overfit_32(golden):
    cfg = golden["overfit"]
    rec = golden["recipe"]
    n = cfg["images"]
    p = synth.mlp_flat_params(DIMS).astype(np.float64)
    v = np.zeros_like(p)
    X = synth.images_u8(n).astype(np.float64) / 255.0
    y = synth.labels(n, 10)
    loss = None
    for _ in range(cfg["steps"]):
        loss, p, v, _ = oracle.mlp_train_step(DIMS, p, v, X, y, rec["lr"], rec["momentum"])
    final = _loss(DIMS, p, X, y)
    assert final < cfg["max_loss"], final


def test_train_step_composes_parts(golden):
    rec = golden["recipe"]
    dims = [20, 16, 5]
    p = synth.mlp_flat_params(dims, seed=3).astype(np.float64)
    v = synth.normal(3, synth.STREAM_GENERIC, p.size) * 1e-3
    X = synth.images_u8(8, 20, seed=3).astype(np.float64) / 255.0
    y = synth.labels(8, 5, seed=3)
    loss, p1, v1, g = oracle.mlp_train_step(dims, p, v, X, y, rec["lr"], rec["momentum"])
    # the update equals v' = m v - lr g, w' = w + v' for the reported g
    assert np.allclose(v1, rec["momentum"] * v - rec["lr"] * g, rtol=1e-15, atol=1e-18)
    assert np.allclose(p1, p + v1, rtol=1e-15, atol=1e-18)
    assert abs(loss - _loss(dims, p, X, y)) < 1e-15


# ------------------------------------------------------------ block

EPS, SLOPE = 1e-6, 0.5


def _block_inputs(T=5, d=8, h=12, seed=21):
    x = synth.normal(seed, synth.STREAM_BLOCK_X, T * d).reshape(T, d)
    Wg = synth.normal(seed, synth.STREAM_BLOCK_WG, d * h).reshape(d, h) * 0.3
    Wd = synth.normal(seed, synth.STREAM_BLOCK_WD, h * d).reshape(h, d) * 0.3
    dy = synth.normal(seed, synth.STREAM_BLOCK_DY, T * d).reshape(T, d)
    return x, Wg, Wd, dy


def test_block_zero_down_is_identity():
    x, Wg, Wd, dy = _block_inputs()
    y, r = oracle.block_fwd(x, Wg, np.zeros_like(Wd), EPS, SLOPE)
    assert np.array_equal(y, x)
    dx, dWg, dWd = oracle.block_bwd(x, Wg, np.zeros_like(Wd), dy, EPS, SLOPE)
    assert np.array_equal(dx, dy)
    assert np.all(dWg == 0.0)
    assert np.any(dWd != 0.0)


def test_block_zero_gate_is_identity():
    x, Wg, Wd, dy = _block_inputs()
    y, r = oracle.block_fwd(x, np.zeros_like(Wg), Wd, EPS, SLOPE)
    assert np.array_equal(y, x)
    dx, dWg, dWd = oracle.block_bwd(x, np.zeros_like(Wg), Wd, dy, EPS, SLOPE)
    assert np.array_equal(dx, dy)
    assert np.all(dWg == 0.0) and np.all(dWd == 0.0)


def test_block_rstd_constant_rows():
    d = 8
    c = np.array([0.5, -2.0, 1e-4, 3.0])
    x = np.repeat(c[:, None], d, axis=1)
    _, Wg, Wd, _ = _block_inputs(T=4, d=d)
    _, r = oracle.block_fwd(x, Wg, Wd, EPS, SLOPE)
    assert np.allclose(r, 1.0 / np.sqrt(c * c + EPS), rtol=1e-14)


def test_block_single_positive_path_closed_form():
    # d = 1, h = 1: n = x / sqrt(x^2 + eps); u = n wg; y = x + f(u) wd.
    x = np.array([[0.7], [-1.3]])
    for wg in (0.8, -0.8):
        y, _ = oracle.block_fwd(x, np.array([[wg]]), np.array([[0.25]]), EPS, SLOPE)
        n = x / np.sqrt(x * x + EPS)
        u = n * wg
        f = np.where(u > 0, u * u, (SLOPE * u) ** 2)
        assert np.allclose(y, x + 0.25 * f, rtol=1e-14)


def _block_loss(x, Wg, Wd, proj):
    y, _ = oracle.block_fwd(x, Wg, Wd, EPS, SLOPE)
    return float((y * proj).sum())


def test_block_backward_fd():
    x, Wg, Wd, dy = _block_inputs()
    dx, dWg, dWd = oracle.block_bwd(x, Wg, Wd, dy, EPS, SLOPE)
    h = 1e-6
    for arr, grad in ((x, dx), (Wg, dWg), (Wd, dWd)):
        for idx in np.ndindex(arr.shape):
            a0 = arr[idx]
            arr[idx] = a0 + h; lp = _block_loss(x, Wg, Wd, dy)
            arr[idx] = a0 - h; lm = _block_loss(x, Wg, Wd, dy)
            arr[idx] = a0
            fd = (lp - lm) / (2 * h)
            assert abs(grad[idx] - fd) <= 1e-7 + 1e-6 * abs(fd), (idx, grad[idx], fd)


def test_block_sampled_forms_agree():
    x, Wg, Wd, dy = _block_inputs(T=9, d=8, h=12, seed=4)
    x32, Wg32, Wd32, dy32 = (a.astype(np.float32) for a in (x, Wg, Wd, dy))
    xd, Wgd, Wdd, dyd = (a.astype(np.float64) for a in (x32, Wg32, Wd32, dy32))
    y, r = oracle.block_fwd(xd, Wgd, Wdd, EPS, SLOPE)
    dx, dWg, dWd = oracle.block_bwd(xd, Wgd, Wdd, dyd, EPS, SLOPE)
    rows = np.array([8, 1, 3])
    yr, rr = oracle.block_fwd_rows(x32, Wg32, Wd32, rows, EPS, SLOPE)
    assert np.allclose(yr, y[rows], rtol=1e-13, atol=1e-15) and np.allclose(rr, r[rows], rtol=1e-14)
    dxr = oracle.block_bwd_dx_rows(x32, Wg32, Wd32, dy32, rows, EPS, SLOPE)
    assert np.allclose(dxr, dx[rows], rtol=1e-12, atol=1e-14)
    which = np.array([0, 0, 1, 1]); ii = np.array([0, 7, 0, 11]); jj = np.array([11, 3, 7, 0])
    ent = oracle.block_bwd_dw_entries(x32, Wg32, Wd32, dy32, which, ii, jj, EPS, SLOPE)
    want = np.array([dWg[0, 11], dWg[7, 3], dWd[0, 7], dWd[11, 0]])
    assert np.allclose(ent, want, rtol=1e-11, atol=1e-14)


# ------------------------------------------------------------ MSE and stack

def test_mse_closed_forms():
    t = synth.normal(2, synth.STREAM_TARGET, 40)
    L, dy = oracle.mse(t, t)
    assert L == 0.0 and np.all(dy == 0.0)
    L, dy = oracle.mse(t + 0.5, t)
    assert abs(L - 0.25) < 1e-15 and np.allclose(dy, 2 * 0.5 / 40, rtol=1e-14)


def test_stack_fd():
    T, d, h, nb = 4, 6, 10, 2
    x0 = synth.normal(8, synth.STREAM_BLOCK_X, T * d).reshape(T, d)
    tgt = synth.normal(8, synth.STREAM_TARGET, T * d).reshape(T, d)
    params = synth.normal(8, synth.STREAM_BLOCK_WG, nb * 2 * d * h) * 0.3
    loss, g, dx0 = oracle.stack_fwd_bwd(x0, params, nb, d, h, EPS, SLOPE, tgt)

    def L(p, x):
        return oracle.stack_fwd_bwd(x, p, nb, d, h, EPS, SLOPE, tgt)[0]

    hh = 1e-6
    for i in range(params.size):
        pp = params.copy(); pp[i] += hh
        pm = params.copy(); pm[i] -= hh
        fd = (L(pp, x0) - L(pm, x0)) / (2 * hh)
        assert abs(g[i] - fd) <= 1e-8 + 1e-5 * abs(fd), (i, g[i], fd)
    for idx in np.ndindex(x0.shape):
        xp = x0.copy(); xp[idx] += hh
        xm = x0.copy(); xm[idx] -= hh
        fd = (L(params, xp) - L(params, xm)) / (2 * hh)
        assert abs(dx0[idx] - fd) <= 1e-8 + 1e-5 * abs(fd)


# ------------------------------------------------------------ attention preprocessing

def _attn_dims():
    return dict(n_q=2, n_kv=1, hd=64, rope_dims=16, seq_len=5)


def test_attn_prep_rope_closed_form():
    """RMSNorm -> QKV -> QK norm -> partial RoPE -> q gain ("Full-Depth MLP
    Megakernel + Fused Attention Preprocessing", "What Worked" / "What Didn't
    Work") on a case with a closed form: x = ones(4) (r = 1 with eps 0), q head
    u = e_0, k head u = e_1, v head u = 2 e_0.  The QK norm scales a unit
    vector of a 64-wide head to 8; RoPE over R = 4 dims pairs (0, 2) at
    frequency 1 and (1, 3) at frequency theta^(-1/2) = 0.01."""
    d, hd, R = 4, 64, 4
    W = np.zeros((d, 3 * hd))
    W[:, 0] = 0.25             # q dim 0
    W[:, hd + 1] = 0.25        # k dim 1
    W[:, 2 * hd] = 0.5         # v dim 0
    T = 4
    x = np.ones((T, d))
    out = oracle.attn_prep(x, W, np.array([1.5]), 1, 1, hd, R, seq_len=100, eps=0.0)
    for p in range(T):
        q, k, v = out[p, :hd], out[p, hd:2 * hd], out[p, 2 * hd:]
        want_q = np.zeros(hd)
        want_q[0], want_q[2] = 8 * math.cos(p), 8 * math.sin(p)
        want_k = np.zeros(hd)
        want_k[1], want_k[3] = 8 * math.cos(0.01 * p), 8 * math.sin(0.01 * p)
        want_v = np.zeros(hd)
        want_v[0] = 2.0
        assert np.allclose(q, 1.5 * want_q, rtol=0, atol=1e-12)
        assert np.allclose(k, want_k, rtol=0, atol=1e-12)
        assert np.array_equal(v, want_v)


def test_attn_prep_invariants_and_library_special_cases():
    dm = _attn_dims()
    n_q, n_kv, hd = dm["n_q"], dm["n_kv"], dm["hd"]
    T, d = 11, 32
    N = (n_q + 2 * n_kv) * hd
    x = synth.normal(5, synth.STREAM_GENERIC, T * d).reshape(T, d)
    W = synth.normal(5, synth.STREAM_GENERIC + 1, d * N).reshape(d, N) * 0.2
    gain = np.array([0.5, 1.75])
    out = oracle.attn_prep(x, W, gain, eps=0.0, **dm)
    # RMSNorm makes the block invariant to a positive scale of x
    assert np.allclose(oracle.attn_prep(3.0 * x, W, gain, eps=0.0, **dm), out, rtol=1e-12,
                       atol=1e-12)
    # value heads: r (x W)_v, a plain matrix product
    r = 1.0 / np.sqrt((x * x).mean(1))
    u = r[:, None] * (x @ W)
    assert np.allclose(out[:, (n_q + n_kv) * hd:], u[:, (n_q + n_kv) * hd:], rtol=1e-12)
    # RoPE rotates pairs, so every query head keeps RMS |gain| and every key head RMS 1
    for h in range(n_q + n_kv):
        rms = np.sqrt((out[:, h * hd:(h + 1) * hd] ** 2).mean(1))
        assert np.allclose(rms, gain[h] if h < n_q else 1.0, rtol=1e-12)
    # at position 0 (tokens 0 and seq_len) nothing rotates: normalised head x gain
    for t in (0, dm["seq_len"], 2 * dm["seq_len"]):
        for h in range(n_q + n_kv):
            uh = u[t, h * hd:(h + 1) * hd]
            want = uh / np.sqrt((uh * uh).mean()) * (gain[h] if h < n_q else 1.0)
            assert np.allclose(out[t, h * hd:(h + 1) * hd], want, rtol=1e-12)
    # the sampled-rows form (fp32 inputs as stored) agrees with the full form
    rows = np.array([3, 7, 10])
    got = oracle.attn_prep_rows(x.astype(np.float32), W.astype(np.float32), gain, rows, **dm)
    ref = oracle.attn_prep(x.astype(np.float32).astype(np.float64),
                           W.astype(np.float32).astype(np.float64), gain, eps=1e-6, **dm)[rows]
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_rounding_points_modes_round_the_backward_operands():
    """dZ enters the backward matrix multiplies at a rounding point.  With
    identity weights and H = [1, 1], dW2 = H^T dZ; dZ = 1 + 2^-9 survives
    binary16 (fp16 points equal exact mode) but not bf16 (it becomes 1)."""
    dims = [2, 2, 2]
    params = np.zeros(oracle.param_count(dims))
    params[0:4] = [1, 0, 0, 1]
    params[6:10] = [1, 0, 0, 1]
    X = np.array([[1.0, 1.0]])
    dZ = np.array([[1 + 2.0 ** -9, 0.0]])
    grads = {}
    for name in ("exact", "f16", "bf16"):
        hs, _ = oracle.mlp_forward(dims, params, X, points=name)
        grads[name] = oracle.mlp_backward(dims, params, X, hs, dZ, points=name)
    dw2 = lambda g: g[6:10].reshape(2, 2)
    assert dw2(grads["exact"]).tolist() == [[1 + 2.0 ** -9, 0.0], [1 + 2.0 ** -9, 0.0]]
    assert np.array_equal(dw2(grads["f16"]), dw2(grads["exact"]))
    assert dw2(grads["bf16"]).tolist() == [[1.0, 0.0], [1.0, 0.0]]
    # db2 is the column sum of dZ, taken through the same rounding point
    assert grads["f16"][10:12].tolist() == [1 + 2.0 ** -9, 0.0]
    assert grads["bf16"][10:12].tolist() == [1.0, 0.0]
