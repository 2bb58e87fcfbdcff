"""Parity of the MLP block, the MSE loss and the block stack with the oracle.

Block of "Full-Depth MLP Megakernel + Fused Attention Preprocessing" ("What
Worked"): RMSNorm (eps 1e-6, gain 1) -> W_gate -> LeakyReLU(0.5)^2 -> W_down
-> residual, d = 512, hidden 1536, weights N(0, 0.02), x and dy N(0, 1).
"""
import numpy as np
import pytest
import torch

import oracle
import mlp_step_gb300 as M
from mlp_step_gb300 import synth
from helpers import bf16_values, to_dev, rel_to_max

pytestmark = pytest.mark.gpu

EPS, SLOPE, D = 1e-6, 0.5, 512


@pytest.fixture(scope="module", autouse=True)
def _lib():
    M.load()
    yield
    assert M.get_device_status() == M.MLP_OK


def assert_block_delta(out, ref, base, tol=3e-2):
    """The block's contribution (out - base) within tol of its largest magnitude,
    plus the rounding of the stored bf16 output (2^-8 of |ref| covers the
    half-ulp of the final rounding on top of the fp32 value's own error)."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    base = np.asarray(base, dtype=np.float64)
    bound = tol * np.abs(ref - base).max() + 2.0 ** -8 * np.abs(ref)
    err = np.abs(out - ref)
    assert np.all(err <= bound), float((err / np.maximum(bound, 1e-30)).max())


def _inputs(T, h, seed=0):
    x = synth.normal_f32((T, D), synth.STREAM_BLOCK_X + seed)
    wg = synth.normal_f32((D, h), synth.STREAM_BLOCK_WG + seed, std=0.02)
    wd = synth.normal_f32((h, D), synth.STREAM_BLOCK_WD + seed, std=0.02)
    dy = synth.normal_f32((T, D), synth.STREAM_BLOCK_DY + seed)
    # the values the GPU receives (bf16), as float32
    return tuple(bf16_values(a).astype(np.float32) for a in (x, wg, wd, dy))


def _fwd(x, wg, wd):
    T = x.shape[0]
    xd, gd, dd = (to_dev(a, torch.bfloat16) for a in (x, wg, wd))
    y = torch.full((T, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    r = torch.full((T,), float("nan"), device="cuda")
    M.mlp_block_fwd(xd, gd, dd, y, r, eps=EPS, slope=SLOPE)
    return y, r


@pytest.mark.parametrize("T,h", [(300, 1536), (128, 256), (1, 512), (1000, 1536)])
def test_block_fwd_matches_oracle(T, h):
    x, wg, wd, _ = _inputs(T, h)
    y, r = _fwd(x, wg, wd)
    y_ref, r_ref = oracle.block_fwd(x, wg, wd, EPS, SLOPE)
    yg = y.float().cpu().numpy()
    assert np.all(np.isfinite(yg))
    # y itself, and the block's own contribution y - x
    assert rel_to_max(yg, y_ref) <= 1e-2
    assert_block_delta(yg, y_ref, x)
    assert np.allclose(r.cpu().numpy(), r_ref, rtol=1e-5)


def test_block_fwd_zero_weights_is_identity():
    T, h = 257, 1536
    x, wg, wd, _ = _inputs(T, h)
    y, _ = _fwd(x, wg, np.zeros_like(wd))
    assert np.array_equal(y.float().cpu().numpy(), x)
    y, _ = _fwd(x, np.zeros_like(wg), wd)
    assert np.array_equal(y.float().cpu().numpy(), x)


def test_block_fwd_full_size_sampled_rows():
    T, h = 65536, 1536
    x, wg, wd, _ = _inputs(T, h, seed=1)
    y, r = _fwd(x, wg, wd)
    rows = np.concatenate([synth.randint(3, synth.STREAM_GENERIC, 62, T), [0, T - 1]])
    y_ref, r_ref = oracle.block_fwd_rows(x, wg, wd, rows, EPS, SLOPE)
    yg = y.float().cpu().numpy()[rows]
    assert_block_delta(yg, y_ref, x[rows])
    assert np.allclose(r.cpu().numpy()[rows], r_ref, rtol=1e-5)
    # same result when run again (no races between the CTA pair)
    y2, _ = _fwd(x, wg, wd)
    assert torch.equal(y, y2)


def _bwd(x, wg, wd, dy):
    T = x.shape[0]
    h = wg.shape[1]
    xd, gd, dd, dyd = (to_dev(a, torch.bfloat16) for a in (x, wg, wd, dy))
    y = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    r = torch.empty((T,), device="cuda")
    M.mlp_block_fwd(xd, gd, dd, y, r, eps=EPS, slope=SLOPE)
    dx = torch.full((T, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    dwg = torch.full((D, h), float("nan"), device="cuda")
    dwd = torch.full((h, D), float("nan"), device="cuda")
    ws = torch.empty(M.mlp_block_workspace_bytes(T, D, h), dtype=torch.uint8, device="cuda")
    M.mlp_block_bwd(xd, r, gd, dd, dyd, dx, dwg, dwd, ws, eps=EPS, slope=SLOPE)
    return dx.float().cpu().numpy(), dwg.cpu().numpy(), dwd.cpu().numpy()


@pytest.mark.parametrize("T,h", [(300, 1536), (128, 256), (5, 512)])
def test_block_bwd_matches_oracle(T, h):
    x, wg, wd, dy = _inputs(T, h)
    dx, dwg, dwd = _bwd(x, wg, wd, dy)
    dx_ref, dwg_ref, dwd_ref = oracle.block_bwd(x, wg, wd, dy, EPS, SLOPE)
    for got, ref, name in ((dx, dx_ref, "dx"), (dwg, dwg_ref, "dW_gate"),
                           (dwd, dwd_ref, "dW_down")):
        assert np.all(np.isfinite(got)), name
        assert rel_to_max(got, ref) <= 3e-2, (name, rel_to_max(got, ref))
    assert_block_delta(dx, dx_ref, dy)


def test_block_bwd_zero_down_passes_dy_through():
    T, h = 200, 512
    x, wg, wd, dy = _inputs(T, h)
    dx, dwg, dwd = _bwd(x, wg, np.zeros_like(wd), dy)
    assert np.array_equal(dx, dy)
    assert np.all(dwg == 0.0)


def test_block_bwd_full_size_sampled():
    T, h = 65536, 1536
    x, wg, wd, dy = _inputs(T, h, seed=2)
    dx, dwg, dwd = _bwd(x, wg, wd, dy)
    rows = np.concatenate([synth.randint(5, synth.STREAM_GENERIC, 30, T), [0, T - 1]])
    dx_ref = oracle.block_bwd_dx_rows(x, wg, wd, dy, rows, EPS, SLOPE)
    assert rel_to_max(dx[rows], dx_ref) <= 3e-2
    assert_block_delta(dx[rows], dx_ref, dy[rows])
    n = 24
    which = np.array([0] * (n // 2) + [1] * (n // 2))
    ii = np.where(which == 0, synth.randint(6, synth.STREAM_GENERIC, n, D),
                  synth.randint(6, synth.STREAM_GENERIC, n, h))
    jj = np.where(which == 0, synth.randint(7, synth.STREAM_GENERIC, n, h),
                  synth.randint(7, synth.STREAM_GENERIC, n, D))
    ent = oracle.block_bwd_dw_entries(x, wg, wd, dy, which, ii, jj, EPS, SLOPE)
    got = np.where(which == 0, dwg[ii % D, jj % h], dwd[ii % h, jj % D])
    # sampled entries: relative to the largest sampled magnitude of each matrix
    for w in (0, 1):
        sel = which == w
        assert rel_to_max(got[sel], ent[sel]) <= 3e-2, w


# ------------------------------------------------------------------ MSE

@pytest.mark.parametrize("n", [512 * 300, 1001, 7])
def test_mse_matches_oracle(n):
    y = bf16_values(synth.normal_f32((n,), synth.STREAM_BLOCK_X))
    t = bf16_values(synth.normal_f32((n,), synth.STREAM_TARGET))
    yd, td = to_dev(y.astype(np.float32), torch.bfloat16), to_dev(t.astype(np.float32),
                                                                   torch.bfloat16)
    loss = torch.zeros(4, device="cuda")
    dy = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(M.mse_workspace_bytes(n), dtype=torch.uint8, device="cuda")
    M.mse_loss_fwd_bwd(yd, td, loss, dy, ws)
    L, dy_ref = oracle.mse(y, t)
    assert abs(loss[0].item() - L) <= 1e-5 * L
    assert rel_to_max(dy.float().cpu().numpy(), dy_ref) <= 4e-3


# ------------------------------------------------------------------ stack

def test_stack_step_matches_oracle_small():
    nb, T, h = 2, 256, 256
    x0 = bf16_values(synth.normal_f32((T, D), synth.STREAM_BLOCK_X)).astype(np.float32)
    tgt = bf16_values(synth.normal_f32((T, D), synth.STREAM_TARGET)).astype(np.float32)
    P = M.mlp_stack_param_count(nb, D, h)
    p0 = (synth.normal_f32((P,), synth.STREAM_BLOCK_WG, std=0.02))
    p0 = bf16_values(p0).astype(np.float32)   # master weights start exactly representable
    params = to_dev(p0)
    vel = torch.zeros_like(params)
    grads = torch.zeros_like(params)
    shadow = params.to(torch.bfloat16)
    ws = torch.empty(M.mlp_stack_workspace_bytes(nb, T, D, h), dtype=torch.uint8, device="cuda")
    loss = torch.zeros(4, device="cuda")
    lr, mom = 0.02, 0.95
    M.mlp_stack_train_step(nb, T, D, h, to_dev(x0, torch.bfloat16), to_dev(tgt, torch.bfloat16),
                           params, vel, grads, shadow, lr, mom, loss, ws, eps=EPS, slope=SLOPE)
    L_ref, g_ref, _ = oracle.stack_fwd_bwd(x0, p0, nb, D, h, EPS, SLOPE, tgt)
    assert abs(loss[0].item() - L_ref) <= 1e-3 * L_ref
    g = grads.cpu().numpy()
    per = 2 * D * h
    for b in range(nb):
        for part, sl in (("gate", slice(b * per, b * per + D * h)),
                         ("down", slice(b * per + D * h, (b + 1) * per))):
            assert rel_to_max(g[sl], g_ref[sl]) <= 3e-2, (b, part, rel_to_max(g[sl], g_ref[sl]))
    # one momentum step from zero velocity: w1 = w0 - lr g
    assert torch.allclose(params, to_dev(p0) - lr * grads, rtol=0, atol=1e-6)
    assert torch.equal(shadow, params.to(torch.bfloat16))


def test_stack_eleven_blocks_matches_oracle():
    """The 11-block stack over 6,144 tokens, the smallest token count at which
    every kernel of the 262,144-token step runs in the same form: CTA-pair
    forward, backward-activation and input-gradient kernels, and both
    weight-gradient GEMMs split six ways over the tokens as at full size.
    Loss, every block's W_gate and W_down gradients, the velocity and the
    update against the fp64 oracle's stack and momentum step."""
    nb, T, h = 11, 6144, 1536
    x0 = bf16_values(synth.normal_f32((T, D), synth.STREAM_BLOCK_X)).astype(np.float32)
    tgt = bf16_values(synth.normal_f32((T, D), synth.STREAM_TARGET)).astype(np.float32)
    P = M.mlp_stack_param_count(nb, D, h)
    p0 = bf16_values(synth.normal_f32((P,), synth.STREAM_BLOCK_WG, std=0.02)).astype(np.float32)
    params = to_dev(p0)
    vel = torch.zeros_like(params)
    grads = torch.zeros_like(params)
    shadow = params.to(torch.bfloat16)
    ws = torch.empty(M.mlp_stack_workspace_bytes(nb, T, D, h), dtype=torch.uint8, device="cuda")
    loss = torch.zeros(4, device="cuda")
    lr, mom = 0.02, 0.95
    M.mlp_stack_train_step(nb, T, D, h, to_dev(x0, torch.bfloat16), to_dev(tgt, torch.bfloat16),
                           params, vel, grads, shadow, lr, mom, loss, ws, eps=EPS, slope=SLOPE)
    torch.cuda.synchronize()
    L_ref, g_ref, _ = oracle.stack_fwd_bwd(x0, p0, nb, D, h, EPS, SLOPE, tgt)
    w_ref, v_ref = oracle.sgd_momentum(p0, g_ref, np.zeros(P), lr, mom)
    assert abs(loss[0].item() - L_ref) <= 1e-3, (loss[0].item(), L_ref)
    g = grads.cpu().numpy()
    v = vel.cpu().numpy()
    dw = params.cpu().numpy().astype(np.float64) - p0
    per = 2 * D * h
    for b in range(nb):
        for part, sl in (("gate", slice(b * per, b * per + D * h)),
                         ("down", slice(b * per + D * h, (b + 1) * per))):
            assert rel_to_max(g[sl], g_ref[sl]) <= 3e-2, (b, part, rel_to_max(g[sl], g_ref[sl]))
            assert rel_to_max(v[sl], v_ref[sl]) <= 3e-2, (b, part, "velocity")
            assert rel_to_max(dw[sl], w_ref[sl] - p0[sl]) <= 3e-2, (b, part, "update")
    assert torch.equal(shadow, params.to(torch.bfloat16))


def test_stack_full_size_runs_finite():
    nb, T, h = 11, 262144, 1536
    P = M.mlp_stack_param_count(nb, D, h)
    assert P == 17_301_504
    x0 = to_dev(synth.normal_f32((T, D), synth.STREAM_BLOCK_X), torch.bfloat16)
    tgt = to_dev(synth.normal_f32((T, D), synth.STREAM_TARGET), torch.bfloat16)
    params = to_dev(synth.normal_f32((P,), synth.STREAM_BLOCK_WG, std=0.02))
    vel = torch.zeros_like(params)
    grads = torch.zeros_like(params)
    shadow = params.to(torch.bfloat16)
    ws = torch.empty(M.mlp_stack_workspace_bytes(nb, T, D, h), dtype=torch.uint8, device="cuda")
    loss = torch.zeros(4, device="cuda")
    M.mlp_stack_train_step(nb, T, D, h, x0, tgt, params, vel, grads, shadow, 0.02, 0.95, loss,
                           ws, eps=EPS, slope=SLOPE)
    torch.cuda.synchronize()
    assert np.isfinite(loss[0].item()) and loss[0].item() > 0
    assert torch.isfinite(grads).all()
    assert torch.equal(shadow, params.to(torch.bfloat16))
