"""The wide MLP 1024-8192-8192-1000 at batch 16,384 (bf16 operands, fp32 master
weights), checked at full size on sampled outputs the oracle computes one by
one, and its GEMM shapes checked as single kernels."""
import numpy as np
import pytest
import torch

import oracle
import mlp_step_gb300 as M
from mlp_step_gb300 import synth
from helpers import bf16_values, to_dev, rel_to_max, assert_elementwise

pytestmark = pytest.mark.gpu

DIMS = [1024, 8192, 8192, 1000]
B = 16384


@pytest.fixture(scope="module", autouse=True)
def _lib():
    M.load()
    yield
    assert M.get_device_status() == M.MLP_OK


def _sample_idx(M_, N, n=192, seed=0):
    ii = np.concatenate([synth.randint(seed, synth.STREAM_GENERIC + 20, n, M_), [0, M_ - 1]])
    jj = np.concatenate([synth.randint(seed, synth.STREAM_GENERIC + 21, n, N), [N - 1, 0]])
    return ii, jj


# (M, N, K, a_trans, b_trans, mask, out_bf16): every GEMM shape of the wide step
SHAPES = {
    "fwd2_relu": (16384, 8192, 8192, 0, 0, False, True),
    "fwd3_logits": (16384, 1000, 8192, 0, 0, False, False),
    "dH1_mask": (16384, 8192, 8192, 0, 1, True, True),
    "dH2_k1000": (16384, 8192, 1000, 0, 1, True, True),
    "dW2": (8192, 8192, 16384, 1, 0, False, False),
    "dW3_n1000": (8192, 1000, 16384, 1, 0, False, False),
    "dW1": (1024, 8192, 16384, 1, 0, False, False),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_wide_gemm_shapes_sampled(name):
    M_, N, K, a_t, b_t, mask, out_bf16 = SHAPES[name]
    A = bf16_values(synth.uniform_f32((K, M_) if a_t else (M_, K), synth.STREAM_GENERIC + 1))
    Bm = bf16_values(synth.uniform_f32((N, K) if b_t else (K, N), synth.STREAM_GENERIC + 2))
    A = A.astype(np.float32)
    Bm = Bm.astype(np.float32)
    Ad, Bd = to_dev(A, torch.bfloat16), to_dev(Bm, torch.bfloat16)
    mk = None
    if mask:
        mk = to_dev(synth.uniform_f32((M_, N), synth.STREAM_GENERIC + 3), torch.bfloat16)
    C = torch.full((M_, N), float("nan"), dtype=torch.bfloat16 if out_bf16 else torch.float32,
                   device="cuda")
    M.mlp_gemm(Ad, Bd, C, M_, N, K, a_trans=a_t, b_trans=b_t, mask=mk)
    ii, jj = _sample_idx(M_, N)
    ref = oracle.matmul_entries(A, Bm, ii, jj, a_t=bool(a_t), b_t=bool(b_t))
    if mask:
        ref = np.where(mk.float().cpu().numpy()[ii, jj] > 0, ref, 0.0)
    got = C.float()[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().numpy()
    assert not torch.isnan(C).any(), "unwritten outputs"
    # fp32 accumulation over K terms: rounding grows like sqrt(K) unit roundoffs
    tol = 8e-3 if out_bf16 else max(1e-5, 4e-7 * np.sqrt(K))
    assert rel_to_max(got, ref) <= tol, rel_to_max(got, ref)


@pytest.mark.parametrize("prec", ["bf16", "f16"])
def test_wide_train_step_full_size(prec):
    """The bench's wide step (batch 16,384) with bf16 operands and with the
    fp16 variant ("The Debugging Lesson Was Numerical"), each against the
    oracle rounding at the same points in its format."""
    lr, mom = 0.01, 0.9
    p0 = synth.mlp_flat_params(DIMS)
    X = synth.normal_f32((B, DIMS[0]), synth.STREAM_X)
    y = synth.labels(B, DIMS[-1])
    h16 = torch.float16 if prec == "f16" else torch.bfloat16
    net = M.MLP(DIMS, prec=M.MLP_PREC_FP16 if prec == "f16" else M.MLP_PREC_BF16, max_batch=B,
                params=torch.from_numpy(p0))
    Xd = to_dev(X, h16)
    yd = to_dev(y)
    # forward logits on sampled rows against the oracle (rounding points of the format)
    logits = torch.empty(B, DIMS[-1], device="cuda")
    net.forward(Xd, logits)
    rows = np.concatenate([synth.randint(1, synth.STREAM_GENERIC, 14, B), [0, B - 1]])
    Xb = Xd.float().cpu().numpy()
    Z_ref = oracle.mlp_forward_rows(DIMS, p0, Xb, rows, points=prec)
    assert rel_to_max(logits.cpu().numpy()[rows], Z_ref) <= 3e-2
    # full step: loss is the mean of the per-row losses of those logits
    loss = torch.zeros(4, device="cuda")
    net.train_step(Xd, yd, lr, mom, loss_out=loss)
    torch.cuda.synchronize()
    ws = torch.empty(M.softmax_xent_workspace_bytes(B, DIMS[-1]), dtype=torch.uint8,
                     device="cuda")
    l2 = torch.zeros(4, device="cuda")
    M.softmax_xent_fwd_bwd(logits, yd, l2, workspace=ws)
    assert abs(loss[0].item() - l2[0].item()) <= 1e-6 * abs(l2[0].item())
    assert np.isfinite(loss[0].item())
    g = net.grads
    assert torch.isfinite(g).all()
    # momentum step from zero velocity: w1 = w0 - lr g, v1 = -lr g
    w0 = torch.from_numpy(p0).cuda()
    assert torch.allclose(net.velocity, -lr * g, rtol=1e-6, atol=0)
    assert torch.allclose(net.params, w0 + net.velocity, rtol=0, atol=1e-7)
