"""Parity of the whole MLP training step (through the C ABI) with the fp64 oracle.

The 784-256-10 network of "Capstone 5: train a network with your CUDA
kernels" ("The minimum model": batch 128, lr 0.1, momentum 0.9, seed
20260829), on the fp32 SIMT path and on the bf16 tensor-core path.
"""
import numpy as np
import pytest
import torch

import oracle
import mlp_step_gb300 as M
from mlp_step_gb300 import synth
from helpers import bf16_values, f16_values, to_dev, rel_to_max, assert_elementwise, near_tie_rows

pytestmark = pytest.mark.gpu

DIMS = [784, 256, 10]
LR, MOM = 0.1, 0.9


@pytest.fixture(scope="module", autouse=True)
def _lib():
    M.load()
    yield
    assert M.get_device_status() == M.MLP_OK


def _x_values(xb):
    return xb.astype(np.float32) / np.float32(255)   # what the byte input means


def _segments(dims, flat):
    out, off = [], 0
    for l in range(len(dims) - 1):
        n = dims[l] * dims[l + 1]
        out.append(("W%d" % (l + 1), flat[off:off + n]))
        off += n
        out.append(("b%d" % (l + 1), flat[off:off + dims[l + 1]]))
        off += dims[l + 1]
    return out


@pytest.mark.parametrize("B", [128, 112, 1])
def test_fp32_step_matches_oracle(B):
    p0 = synth.mlp_flat_params(DIMS)
    xb = synth.images_u8(B, 784)
    y = synth.labels(B, 10)
    net = M.MLP(DIMS, prec=M.MLP_PREC_FP32, max_batch=128, params=torch.from_numpy(p0))
    loss = torch.zeros(1, device="cuda")
    am = torch.empty(B, dtype=torch.int32, device="cuda")
    net.train_step(to_dev(xb), to_dev(y), LR, MOM, loss_out=loss, argmax_out=am)
    torch.cuda.synchronize()
    X = _x_values(xb).astype(np.float64)
    l_ref, p_ref, v_ref, g_ref = oracle.mlp_train_step(DIMS, p0.astype(np.float64),
                                                       np.zeros(p0.size), X, y, LR, MOM)
    # weights after one step: max relative error 1e-4 (elementwise, with the
    # 1e-6 floor of the capstone's step bound)
    assert_elementwise(net.params.cpu().numpy(), p_ref, 1e-4, 1e-6, "params")
    assert_elementwise(net.velocity.cpu().numpy(), v_ref, 1e-4, 1e-7, "velocity")
    assert abs(loss.item() - l_ref) <= 1e-5
    # argmax of the step's forward is bit-exact against the oracle
    _, Z = oracle.mlp_forward(DIMS, p0.astype(np.float64), X)
    ok = ~near_tie_rows(Z)
    assert np.array_equal(am.cpu().numpy()[ok], np.argmax(Z, 1)[ok])


def test_fp32_forward_logits_and_backward_grads():
    B = 128
    p0 = synth.mlp_flat_params(DIMS)
    xb = synth.images_u8(B, 784)
    net = M.MLP(DIMS, prec=M.MLP_PREC_FP32, max_batch=B, params=torch.from_numpy(p0))
    X = _x_values(xb)
    logits = torch.empty(B, 10, device="cuda")
    net.forward(to_dev(X), logits)
    hs, Z = oracle.mlp_forward(DIMS, p0.astype(np.float64), X.astype(np.float64))
    assert_elementwise(logits.cpu().numpy(), Z, 1e-4, 1e-5, "logits")
    dZ = synth.normal_f32((B, 10), synth.STREAM_GENERIC, std=0.01)
    dx = torch.empty(B, 784, device="cuda")
    net.backward(to_dev(dZ), B, dx=dx)
    g_ref, dX_ref = oracle.mlp_backward(DIMS, p0.astype(np.float64), X.astype(np.float64), hs,
                                        dZ.astype(np.float64), want_dx=True)
    for (name, got), (_, ref) in zip(_segments(DIMS, net.grads.cpu().numpy()),
                                     _segments(DIMS, g_ref)):
        assert rel_to_max(got, ref) <= 1e-5, name
    assert rel_to_max(dx.cpu().numpy(), dX_ref) <= 1e-5


@pytest.mark.parametrize("B", [128, 112, 1])
def test_bf16_step_matches_oracle(B):
    p0 = synth.mlp_flat_params(DIMS)
    xb = synth.images_u8(B, 784)
    y = synth.labels(B, 10)
    net = M.MLP(DIMS, prec=M.MLP_PREC_BF16, max_batch=128, params=torch.from_numpy(p0))
    loss = torch.zeros(1, device="cuda")
    net.train_step(to_dev(xb), to_dev(y), LR, MOM, loss_out=loss)
    torch.cuda.synchronize()
    Xb = bf16_values(_x_values(xb))
    l_ref, p_ref, v_ref, g_ref = oracle.mlp_train_step(DIMS, p0.astype(np.float64),
                                                       np.zeros(p0.size), Xb, y, LR, MOM,
                                                       bf16_points=True)
    assert abs(loss.item() - l_ref) <= 1e-3
    for (name, got), (_, ref) in zip(_segments(DIMS, net.grads.cpu().numpy()),
                                     _segments(DIMS, g_ref)):
        assert rel_to_max(got, ref) <= 3e-2, name
    assert rel_to_max(net.params.cpu().numpy() - p0, p_ref - p0) <= 3e-2
    # the bf16 shadow is the rounded fp32 master weight
    W1 = net.params[:784 * 256].view(784, 256)
    S1 = net.shadow[:784 * 256].view(784, 256)
    assert torch.equal(S1, W1.to(torch.bfloat16))
    W2 = net.params[200960:200960 + 2560].view(256, 10)
    S2 = net.shadow[784 * 256:].view(256, 16)
    assert torch.equal(S2[:, :10], W2.to(torch.bfloat16))


@pytest.mark.parametrize("B", [128, 112])
def test_f16_step_matches_oracle(B):
    """The fp16-operand variant ("The Debugging Lesson Was Numerical": FP16 in,
    FP32 accumulate) against the oracle rounding at the same points to binary16."""
    p0 = synth.mlp_flat_params(DIMS)
    xb = synth.images_u8(B, 784)
    y = synth.labels(B, 10)
    net = M.MLP(DIMS, prec=M.MLP_PREC_FP16, max_batch=128, params=torch.from_numpy(p0))
    loss = torch.zeros(1, device="cuda")
    am = torch.empty(B, dtype=torch.int32, device="cuda")
    net.train_step(to_dev(xb), to_dev(y), LR, MOM, loss_out=loss, argmax_out=am)
    torch.cuda.synchronize()
    Xh = f16_values(_x_values(xb))
    l_ref, p_ref, v_ref, g_ref = oracle.mlp_train_step(DIMS, p0.astype(np.float64),
                                                       np.zeros(p0.size), Xh, y, LR, MOM,
                                                       points="f16")
    assert abs(loss.item() - l_ref) <= 1e-3
    for (name, got), (_, ref) in zip(_segments(DIMS, net.grads.cpu().numpy()),
                                     _segments(DIMS, g_ref)):
        assert rel_to_max(got, ref) <= 3e-2, name
    assert rel_to_max(net.params.cpu().numpy() - p0, p_ref - p0) <= 3e-2
    # predictions of the step's forward, where the top two logits are apart
    hs, Z = oracle.mlp_forward(DIMS, p0.astype(np.float64), Xh, points="f16")
    ok = ~near_tie_rows(Z, rel=1e-2)
    assert np.array_equal(am.cpu().numpy()[ok], np.argmax(Z, 1)[ok])
    # the fp16 shadow is the rounded fp32 master weight
    W1 = net.params[:784 * 256].view(784, 256)
    S1 = net.shadow[:784 * 256].view(784, 256)
    assert S1.dtype == torch.float16 and torch.equal(S1, W1.to(torch.float16))
    W2 = net.params[200960:200960 + 2560].view(256, 10)
    S2 = net.shadow[784 * 256:].view(256, 16)
    assert torch.equal(S2[:, :10], W2.to(torch.float16))


def test_f16_step_matches_unfused_sequence_and_epoch():
    """fp16 networks run the same step program; the separate calls (forward,
    loss with fp16 dZ, backward, SGD) give the same step, and an epoch equals
    its steps in sequence bit for bit."""
    B, n = 128, 3 * 128 + 40
    p0 = synth.mlp_flat_params(DIMS)
    p0[200704:200960] = synth.normal_f32((256,), synth.STREAM_GENERIC, std=0.1)  # nonzero b1
    xb = to_dev(synth.images_u8(n, 784))
    y = to_dev(synth.labels(n, 10))
    fused = M.MLP(DIMS, prec=M.MLP_PREC_FP16, max_batch=B, params=torch.from_numpy(p0))
    loss_f = torch.zeros(4, device="cuda")
    for _ in range(2):
        fused.train_step(xb[:B], y[:B], LR, MOM, loss_out=loss_f)
    seq = M.MLP(DIMS, prec=M.MLP_PREC_FP16, max_batch=B, params=torch.from_numpy(p0))
    logits = torch.empty(B, 10, device="cuda")
    dl = torch.empty(B, 16, dtype=torch.float16, device="cuda")
    loss_s = torch.zeros(4, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        seq.forward(xb[:B], logits)
        M.softmax_xent_fwd_bwd(logits, y[:B], loss_s, dlogits=dl, workspace=ws)
        seq.backward(dl, B)
        seq.sgd_step(LR, MOM)
    torch.cuda.synchronize()
    assert abs(loss_f[0].item() - loss_s[0].item()) <= 1e-6 * abs(loss_s[0].item())
    assert torch.allclose(fused.grads, seq.grads, rtol=1e-5, atol=1e-9)
    assert torch.allclose(fused.params, seq.params, rtol=1e-6, atol=1e-8)
    ep = M.MLP(DIMS, prec=M.MLP_PREC_FP16, max_batch=B, params=torch.from_numpy(p0))
    losses = torch.zeros(4, device="cuda")
    ep.train_epoch(xb, y, LR, MOM, B, losses_out=losses)
    sq = M.MLP(DIMS, prec=M.MLP_PREC_FP16, max_batch=B, params=torch.from_numpy(p0))
    loss_q = torch.zeros(4, 4, device="cuda")
    for s_ in range(4):
        a, b = s_ * B, min(n, (s_ + 1) * B)
        sq.train_step(xb[a:b], y[a:b], LR, MOM, loss_out=loss_q[s_])
    torch.cuda.synchronize()
    assert torch.equal(losses, loss_q[:, 0])
    for name in ("params", "velocity", "grads", "shadow"):
        assert torch.equal(getattr(ep, name), getattr(sq, name)), name
    assert M.get_device_status() == M.MLP_OK


def test_bf16_fused_step_matches_unfused_sequence():
    """The train step fuses softmax cross entropy into the logits GEMM and the
    momentum update into the weight-gradient GEMMs; the separate calls
    (forward, loss, backward, SGD) must give the same step."""
    B = 128
    p0 = synth.mlp_flat_params(DIMS)
    p0[200704:200960] = synth.normal_f32((256,), synth.STREAM_GENERIC, std=0.1)  # nonzero b1
    xb = to_dev(synth.images_u8(B, 784))
    y = to_dev(synth.labels(B, 10))
    fused = M.MLP(DIMS, prec=M.MLP_PREC_BF16, max_batch=B, params=torch.from_numpy(p0))
    loss_f = torch.zeros(4, device="cuda")
    am_f = torch.empty(B, dtype=torch.int32, device="cuda")
    for _ in range(2):   # second step also exercises a nonzero velocity
        fused.train_step(xb, y, LR, MOM, loss_out=loss_f, argmax_out=am_f)
    seq = M.MLP(DIMS, prec=M.MLP_PREC_BF16, max_batch=B, params=torch.from_numpy(p0))
    logits = torch.empty(B, 10, device="cuda")
    dl = torch.empty(B, 16, dtype=torch.bfloat16, device="cuda")
    loss_s = torch.zeros(4, device="cuda")
    am_s = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        seq.forward(xb, logits)
        M.softmax_xent_fwd_bwd(logits, y, loss_s, dlogits=dl, argmax_out=am_s, workspace=ws)
        seq.backward(dl, B)
        seq.sgd_step(LR, MOM)
    torch.cuda.synchronize()
    assert abs(loss_f[0].item() - loss_s[0].item()) <= 1e-6 * abs(loss_s[0].item())
    assert torch.equal(am_f, am_s)
    assert torch.allclose(fused.grads, seq.grads, rtol=1e-5, atol=1e-9)
    assert torch.allclose(fused.params, seq.params, rtol=1e-6, atol=1e-8)
    assert torch.allclose(fused.velocity, seq.velocity, rtol=1e-5, atol=1e-9)
    assert torch.equal(fused.shadow, seq.shadow) or \
        (fused.shadow.float() - seq.shadow.float()).abs().max().item() <= 2 ** -7


def test_bf16_epoch_matches_step_sequence():
    """mlp_train_epoch runs the full-size steps as one launch (a grid barrier
    between steps) and the remainder as an ordinary step: every result must
    equal the step-by-step sequence bit for bit."""
    B, n = 128, 3 * 128 + 40
    p0 = synth.mlp_flat_params(DIMS)
    xb = to_dev(synth.images_u8(n, 784))
    y = to_dev(synth.labels(n, 10))
    ep = M.MLP(DIMS, prec=M.MLP_PREC_BF16, max_batch=B, params=torch.from_numpy(p0))
    losses = torch.zeros(4, device="cuda")
    am_e = torch.empty(n, dtype=torch.int32, device="cuda")
    ep.train_epoch(xb, y, LR, MOM, B, losses_out=losses, argmax_out=am_e)
    sq = M.MLP(DIMS, prec=M.MLP_PREC_BF16, max_batch=B, params=torch.from_numpy(p0))
    loss_s = torch.zeros(4, 4, device="cuda")
    am_s = torch.empty(n, dtype=torch.int32, device="cuda")
    for s in range(4):
        a, b = s * B, min(n, (s + 1) * B)
        sq.train_step(xb[a:b], y[a:b], LR, MOM, loss_out=loss_s[s], argmax_out=am_s[a:b])
    torch.cuda.synchronize()
    assert torch.equal(losses, loss_s[:, 0])
    assert torch.equal(am_e, am_s)
    for name in ("params", "velocity", "grads", "shadow"):
        assert torch.equal(getattr(ep, name), getattr(sq, name)), name
    assert M.get_device_status() == M.MLP_OK


def _oracle_epoch(p0, X, y, B, perturb=0.0):
    """Losses and final parameters of the oracle's epoch at the bf16 points,
    the velocity carried from step to step; perturb scales the starting
    weights by (1 + perturb * n_i) with n_i ~ N(0, 1) drawn once."""
    p = p0.astype(np.float64)
    if perturb:
        p = p * (1.0 + perturb * synth.normal(9, synth.STREAM_GENERIC + 61, p.size))
    v = np.zeros(p.size)
    losses = []
    for s in range((len(y) + B - 1) // B):
        a, b = s * B, min(len(y), (s + 1) * B)
        l, p, v, _ = oracle.mlp_train_step(DIMS, p, v, X[a:b], y[a:b], LR, MOM, bf16_points=True)
        losses.append(l)
    return np.array(losses), p


def test_bf16_epoch_trajectory_matches_oracle():
    """One epoch of 6,000 images ("Capstone 5", "Checked results, after the
    prediction": 46 steps of batch 128 and one of 112, lr 0.1, momentum 0.9).

    * Step by step: each of the 47 steps, run through the library, against the
      oracle step (bf16 rounding points) started from the library's own
      parameters and velocity before that step: loss within 1e-3, the update
      and the new velocity within 3e-2 of their largest entry per tensor.
    * mlp_train_epoch (all full steps in one launch) equals that step
      sequence bit for bit.
    * Free-running: the epoch against the oracle's own epoch.  At the bf16
      points the method amplifies tiny changes of the weights (a 16-bit
      rounding flips; measured: a 2^-24 relative change of the starting
      weights moves the oracle's own loss by up to about 1e-2 within the
      epoch), so the losses and the weights' change over the epoch are held
      to 1e-3 (3e-2) plus four times that spread, measured here."""
    B, n = 128, 6000
    p0 = synth.mlp_flat_params(DIMS)
    xb = synth.images_u8(n, 784)
    y = synth.labels(n, 10)
    X = bf16_values(_x_values(xb))
    xd, yd = to_dev(xb), to_dev(y)
    n_steps = (n + B - 1) // B
    # the step sequence, state before every step kept
    sq = M.MLP(DIMS, prec=M.MLP_PREC_BF16, max_batch=B, params=torch.from_numpy(p0))
    loss_s = torch.zeros(n_steps, 4, device="cuda")
    states = []
    for s in range(n_steps):
        states.append((sq.params.double().cpu().numpy(), sq.velocity.double().cpu().numpy()))
        a, b = s * B, min(n, (s + 1) * B)
        sq.train_step(xd[a:b], yd[a:b], LR, MOM, loss_out=loss_s[s])
    torch.cuda.synchronize()
    states.append((sq.params.double().cpu().numpy(), sq.velocity.double().cpu().numpy()))
    got_losses = loss_s[:, 0].double().cpu().numpy()
    for s in range(n_steps):
        a, b = s * B, min(n, (s + 1) * B)
        (p_s, v_s), (p_n, v_n) = states[s], states[s + 1]
        l_ref, p_ref, v_ref, _ = oracle.mlp_train_step(DIMS, p_s, v_s, X[a:b], y[a:b], LR, MOM,
                                                       bf16_points=True)
        assert abs(got_losses[s] - l_ref) <= 1e-3, (s, got_losses[s], l_ref)
        for (name, g), (_, r) in zip(_segments(DIMS, p_n - p_s), _segments(DIMS, p_ref - p_s)):
            assert rel_to_max(g, r) <= 3e-2, (s, "update", name, rel_to_max(g, r))
        for (name, g), (_, r) in zip(_segments(DIMS, v_n), _segments(DIMS, v_ref)):
            assert rel_to_max(g, r) <= 3e-2, (s, "velocity", name)
    # the epoch call: bit for bit the step sequence
    ep = M.MLP(DIMS, prec=M.MLP_PREC_BF16, max_batch=B, params=torch.from_numpy(p0))
    losses = torch.full((n_steps,), float("nan"), device="cuda")
    ep.train_epoch(xd, yd, LR, MOM, B, losses_out=losses)
    torch.cuda.synchronize()
    assert torch.equal(losses, loss_s[:, 0])
    for name in ("params", "velocity", "shadow"):
        assert torch.equal(getattr(ep, name), getattr(sq, name)), name
    # free-running, against the oracle's epoch and its own spread
    ref_losses, p_ref = _oracle_epoch(p0, X, y, B)
    pert_losses, p_pert = _oracle_epoch(p0, X, y, B, perturb=2.0 ** -24)
    spread = np.abs(pert_losses - ref_losses).max()
    assert np.abs(got_losses - ref_losses).max() <= 1e-3 + 4 * spread, (
        np.abs(got_losses - ref_losses).max(), spread)
    got = states[-1][0]
    for (name, g), (_, r), (_, rp), (_, w0) in zip(_segments(DIMS, got), _segments(DIMS, p_ref),
                                                   _segments(DIMS, p_pert),
                                                   _segments(DIMS, p0)):
        tol = 3e-2 + 4 * rel_to_max(rp - w0, r - w0)
        assert rel_to_max(g - w0, r - w0) <= tol, (name, rel_to_max(g - w0, r - w0), tol)


def test_nonfinite_loss_is_reported():
    """A step whose loss is not finite returns MLP_OK from the call (the work
    is enqueued) and MLP_ERR_NUMERIC from mlp_get_device_status ("Capstone
    5", "The independent submission gate": exit code zero alone does not
    prove the network is correct); the status is cleared by reading it."""
    B = 128
    p0 = synth.mlp_flat_params(DIMS)
    x = torch.from_numpy(_x_values(synth.images_u8(B, 784))).cuda()
    x[3, 100] = float("inf")
    y = to_dev(synth.labels(B, 10))
    for prec in (M.MLP_PREC_BF16, M.MLP_PREC_FP32):
        net = M.MLP(DIMS, prec=prec, max_batch=B, params=torch.from_numpy(p0))
        loss = torch.zeros(1, device="cuda")
        net.train_step(x, y, LR, MOM, loss_out=loss)
        assert M.get_device_status() == M.MLP_ERR_NUMERIC
        assert not np.isfinite(loss.item())
        assert M.get_device_status() == M.MLP_OK
    # finite inputs leave the status clear
    net = M.MLP(DIMS, prec=M.MLP_PREC_BF16, max_batch=B, params=torch.from_numpy(p0))
    net.train_step(torch.from_numpy(_x_values(synth.images_u8(B, 784))).cuda(), y, LR, MOM)
    assert M.get_device_status() == M.MLP_OK


@pytest.mark.parametrize("rem", [0, 40])
def test_bf16_epochs_with_even_step_counts_match_step_sequence(rem):
    """Epoch programs alternate two input buffers; after an even number of
    full steps the handle's input names the second one.  Two epochs in a row
    (2 full steps each, with or without a remainder) and a forward afterwards
    must still equal the step-by-step sequence bit for bit."""
    B = 128
    n = 2 * B + rem
    p0 = synth.mlp_flat_params(DIMS)
    xb = to_dev(synth.images_u8(2 * n, 784))
    y = to_dev(synth.labels(2 * n, 10))
    ep = M.MLP(DIMS, prec=M.MLP_PREC_BF16, max_batch=B, params=torch.from_numpy(p0))
    sq = M.MLP(DIMS, prec=M.MLP_PREC_BF16, max_batch=B, params=torch.from_numpy(p0))
    steps = (n + B - 1) // B
    losses = torch.zeros(2 * steps, device="cuda")
    loss_s = torch.zeros(2 * steps, 4, device="cuda")
    for e in range(2):
        a0 = e * n
        ep.train_epoch(xb[a0:a0 + n], y[a0:a0 + n], LR, MOM, B,
                       losses_out=losses[e * steps:(e + 1) * steps])
        for s in range(steps):
            a, b = a0 + s * B, a0 + min(n, (s + 1) * B)
            sq.train_step(xb[a:b], y[a:b], LR, MOM, loss_out=loss_s[e * steps + s])
    torch.cuda.synchronize()
    assert torch.equal(losses, loss_s[:, 0])
    for name in ("params", "velocity", "grads", "shadow"):
        assert torch.equal(getattr(ep, name), getattr(sq, name)), name
    # the handle's own input buffer is usable afterwards
    lg_e = torch.empty(B, 10, device="cuda")
    lg_s = torch.empty(B, 10, device="cuda")
    ep.forward(xb[:B], lg_e)
    sq.forward(xb[:B], lg_s)
    torch.cuda.synchronize()
    assert torch.equal(lg_e, lg_s)
    assert M.get_device_status() == M.MLP_OK


def test_bf16_epoch_rejects_misaligned_steps():
    net = M.MLP(DIMS, prec=M.MLP_PREC_BF16, max_batch=128)
    xb = torch.zeros(12, 784, dtype=torch.uint8, device="cuda")
    y = torch.zeros(12, dtype=torch.int32, device="cuda")
    with pytest.raises(M.MlpError) as e:
        net.train_epoch(xb, y, LR, MOM, 6)   # each step's labels would start on 24-byte steps
    assert e.value.status == M.MLP_ERR_MISALIGNED


def test_bf16_three_layer_step_program_matches_unfused_sequence():
    """A three-layer net's step program merges each layer's update into the
    next layer's input-gradient phase; it must equal the separate calls."""
    dims = [200, 96, 48, 10]
    B = 100
    p0 = synth.mlp_flat_params(dims)
    xb = to_dev(synth.normal_f32((B, 200), synth.STREAM_GENERIC + 3))
    y = to_dev(synth.labels(B, 10))
    fused = M.MLP(dims, prec=M.MLP_PREC_BF16, max_batch=B, params=torch.from_numpy(p0))
    loss_f = torch.zeros(4, device="cuda")
    for _ in range(2):
        fused.train_step(xb, y, LR, MOM, loss_out=loss_f)
    seq = M.MLP(dims, prec=M.MLP_PREC_BF16, max_batch=B, params=torch.from_numpy(p0))
    logits = torch.empty(B, 10, device="cuda")
    dl = torch.empty(B, 16, dtype=torch.bfloat16, device="cuda")
    loss_s = torch.zeros(4, device="cuda")
    ws = torch.empty(M.softmax_xent_workspace_bytes(B, 10) + 16, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        seq.forward(xb, logits)
        M.softmax_xent_fwd_bwd(logits, y, loss_s, dlogits=dl, workspace=ws)
        seq.backward(dl, B)
        seq.sgd_step(LR, MOM)
    torch.cuda.synchronize()
    assert abs(loss_f[0].item() - loss_s[0].item()) <= 1e-6 * abs(loss_s[0].item())
    assert torch.allclose(fused.params, seq.params, rtol=1e-6, atol=1e-8)
    assert torch.allclose(fused.velocity, seq.velocity, rtol=1e-5, atol=1e-9)
    # shadow rows of the wider layers are padded to whole 128-byte lines
    # (96 -> 128 and 48 -> 64 columns): each row holds bf16 of the updated
    # weight row, the padding stays zero, through both update paths
    for net in (fused, seq):
        assert_shadow_layout(dims, net)
    assert M.get_device_status() == M.MLP_OK


def assert_shadow_layout(dims, net):
    pitch = lambda n: (n + 7) // 8 * 8 if n <= 16 else (n + 63) // 64 * 64
    assert net.shadow.numel() == sum(dims[l] * pitch(dims[l + 1]) for l in range(len(dims) - 1))
    off = soff = 0
    for l in range(len(dims) - 1):
        fi, fo = dims[l], dims[l + 1]
        W = net.params[off:off + fi * fo].view(fi, fo)
        S = net.shadow[soff:soff + fi * pitch(fo)].view(fi, pitch(fo))
        assert torch.equal(S[:, :fo], W.to(torch.bfloat16)), l
        assert not S[:, fo:].float().abs().any(), l
        off += fi * fo + fo
        soff += fi * pitch(fo)


def test_bf16_forward_matches_oracle_exact_mode():
    B = 128
    p0 = synth.mlp_flat_params(DIMS)
    xb = synth.images_u8(B, 784)
    net = M.MLP(DIMS, prec=M.MLP_PREC_BF16, max_batch=B, params=torch.from_numpy(p0))
    logits = torch.empty(B, 10, device="cuda")
    net.forward(to_dev(xb), logits)
    _, Z = oracle.mlp_forward(DIMS, p0.astype(np.float64), _x_values(xb).astype(np.float64))
    assert rel_to_max(logits.cpu().numpy(), Z) <= 3e-2


def test_bf16_steps_are_deterministic():
    B = 128
    p0 = synth.mlp_flat_params(DIMS)
    xb = to_dev(synth.images_u8(B, 784))
    y = to_dev(synth.labels(B, 10))
    outs = []
    for _ in range(2):
        net = M.MLP(DIMS, prec=M.MLP_PREC_BF16, max_batch=B, params=torch.from_numpy(p0))
        for _ in range(3):
            net.train_step(xb, y, LR, MOM)
        outs.append(net.params.clone())
    assert torch.equal(outs[0], outs[1])


def test_overfit_32_on_gpu():
    # "Stage 3: prove that it learns": 32 images, 200 steps, loss below 0.01.
    n = 32
    p0 = synth.mlp_flat_params(DIMS)
    xb = to_dev(synth.images_u8(n, 784))
    y = to_dev(synth.labels(n, 10))
    for prec in (M.MLP_PREC_FP32, M.MLP_PREC_BF16):
        net = M.MLP(DIMS, prec=prec, max_batch=n, params=torch.from_numpy(p0))
        loss = torch.zeros(1, device="cuda")
        for _ in range(200):
            net.train_step(xb, y, LR, MOM, loss_out=loss)
        logits = torch.empty(n, 10, device="cuda")
        net.forward(xb, logits)
        ws = torch.empty(16, dtype=torch.uint8, device="cuda")
        final = torch.zeros(1, device="cuda")
        M.softmax_xent_fwd_bwd(logits, y, final, workspace=ws)
        assert final.item() < 0.01, (prec, final.item())


def test_fp32_forward_backward_linear_order_is_bit_exact():
    """In MLP_ORDER_LINEAR the fp32 path's forward logits and backward
    gradients are chains of fp32 fused multiply-adds in ascending order, so
    the oracle's linear-order GEMMs composed layer by layer give them to the
    bit ("HIP + Vulkan backends -- Phase 3": bit parity through linear-order
    sums)."""
    B = 128
    p0 = synth.mlp_flat_params(DIMS)
    p0[200704:200960] = synth.normal_f32((256,), synth.STREAM_GENERIC, std=0.1)  # nonzero b1
    xb = synth.images_u8(B, 784)
    dZ = synth.normal_f32((B, 10), synth.STREAM_GENERIC + 3, std=0.01)
    M.set_reduction_order(M.MLP_ORDER_LINEAR)
    try:
        net = M.MLP(DIMS, prec=M.MLP_PREC_FP32, max_batch=B, params=torch.from_numpy(p0))
        logits = torch.empty(B, 10, device="cuda")
        net.forward(to_dev(xb), logits)
        net.backward(to_dev(dZ), B)
        torch.cuda.synchronize()
    finally:
        M.set_reduction_order(M.MLP_ORDER_FAST)
    X = _x_values(xb)
    W1, b1 = p0[:200704].reshape(784, 256), p0[200704:200960]
    W2, b2 = p0[200960:203520].reshape(256, 10), p0[203520:]
    H = oracle.matmul_f32_linear(X, W1, bias=b1, act=1)
    Z = oracle.matmul_f32_linear(H, W2, bias=b2)
    assert np.array_equal(logits.cpu().numpy(), Z)
    ones = np.ones((B, 1), dtype=np.float32)
    g2 = oracle.matmul_f32_linear(np.hstack([H, ones]), dZ, a_t=1)          # [dW2; db2]
    dH = oracle.matmul_f32_linear(dZ, W2, b_t=1, mask=H)                      # (dZ W2^T) * (H > 0)
    g1 = oracle.matmul_f32_linear(np.hstack([X, ones]), dH, a_t=1)          # [dW1; db1]
    g = net.grads.cpu().numpy()
    assert np.array_equal(g[:200960].reshape(785, 256), g1)
    assert np.array_equal(g[200960:].reshape(257, 10), g2)
