"""The wide MLP 1024-8192-8192-1000 (bf16 operands, fp32 master weights): the
whole step against the oracle at batch 3,072 (the same kernel for every GEMM
as at 16,384), the 16,384 step on sampled outputs the oracle computes one by
one, and every GEMM shape of the 16,384 step as a single kernel."""
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


# (M, N, K, a_trans, b_trans, mask, out_bf16): every GEMM shape of the wide step;
# the step's weight-gradient GEMMs run over [In | 1] (a ones column after the
# layer input, row pitch rounded up to 64) and produce [dW; db] with M = in + 1
SHAPES = {
    "fwd2_relu": (16384, 8192, 8192, 0, 0, False, True),
    "fwd3_logits": (16384, 1000, 8192, 0, 0, False, False),
    "dH1_mask": (16384, 8192, 8192, 0, 1, True, True),
    "dH2_k1000": (16384, 8192, 1000, 0, 1, True, True),
    "dW2": (8192, 8192, 16384, 1, 0, False, False),
    "dW3_n1000": (8192, 1000, 16384, 1, 0, False, False),
    "dW1": (1024, 8192, 16384, 1, 0, False, False),
    "dW2_ones_row": (8193, 8192, 16384, 1, 0, False, False),
    "dW1_ones_row": (1025, 8192, 16384, 1, 0, False, False),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_wide_gemm_shapes_sampled(name):
    M_, N, K, a_t, b_t, mask, out_bf16 = SHAPES[name]
    A = bf16_values(synth.uniform_f32((K, M_) if a_t else (M_, K), synth.STREAM_GENERIC + 1))
    Bm = bf16_values(synth.uniform_f32((N, K) if b_t else (K, N), synth.STREAM_GENERIC + 2))
    A = A.astype(np.float32)
    Bm = Bm.astype(np.float32)
    Ad, Bd = to_dev(A, torch.bfloat16), to_dev(Bm, torch.bfloat16)
    if a_t and M_ % 8:
        # rows of [In | 1] padded to whole 128-byte lines, as the step stores them
        pitch = (M_ + 63) // 64 * 64
        Ap = torch.zeros(K, pitch, dtype=torch.bfloat16, device="cuda")
        Ap[:, :M_] = Ad
        Ad = Ap[:, :M_]
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


def _wide_segments(flat):
    out, off = [], 0
    for l in range(len(DIMS) - 1):
        n = DIMS[l] * DIMS[l + 1]
        out.append(("W%d" % (l + 1), flat[off:off + n]))
        off += n
        out.append(("b%d" % (l + 1), flat[off:off + DIMS[l + 1]]))
        off += DIMS[l + 1]
    return out


def test_wide_train_step_full_path_matches_oracle():
    """The whole wide step at batch 3,072, the smallest batch at which every
    GEMM takes the kernel it takes at 16,384: CTA-pair tiles without split-K
    for the forward and input-gradient GEMMs (the 1000-wide logits included),
    single-CTA tiles for [dW1; db1] (M = 1025) and pair tiles for [dW2; db2]
    and [dW3; db3] (M = 8193), and the 1000-class loss with its padded bf16
    dZ.  Loss, every weight and bias gradient, the velocity and the update
    against the oracle step rounding at the bf16 points ("Capstone 5",
    "Stage 2: backward and update": every gradient against the float64
    result)."""
    Bsz, lr, mom = 3072, 0.01, 0.9
    p0 = synth.mlp_flat_params(DIMS)
    X = synth.normal_f32((Bsz, DIMS[0]), synth.STREAM_X)
    y = synth.labels(Bsz, DIMS[-1])
    net = M.MLP(DIMS, prec=M.MLP_PREC_BF16, max_batch=Bsz, params=torch.from_numpy(p0))
    Xd = to_dev(X, torch.bfloat16)
    loss = torch.zeros(4, device="cuda")
    net.train_step(Xd, to_dev(y), lr, mom, loss_out=loss)
    torch.cuda.synchronize()
    assert M.get_device_status() == M.MLP_OK
    Xb = Xd.double().cpu().numpy()
    l_ref, p_ref, v_ref, g_ref = oracle.mlp_train_step(DIMS, p0.astype(np.float64),
                                                       np.zeros(p0.size), Xb, y, lr, mom,
                                                       points="bf16")
    assert abs(loss[0].item() - l_ref) <= 1e-3, (loss[0].item(), l_ref)
    g = net.grads.cpu().numpy()
    v = net.velocity.cpu().numpy()
    dp = net.params.cpu().numpy() - p0
    for (name, a), (_, b) in zip(_wide_segments(g), _wide_segments(g_ref)):
        assert rel_to_max(a, b) <= 3e-2, (name, rel_to_max(a, b))
    for (name, a), (_, b) in zip(_wide_segments(v), _wide_segments(v_ref)):
        assert rel_to_max(a, b) <= 3e-2, ("velocity", name)
    for (name, a), (_, b) in zip(_wide_segments(dp), _wide_segments(p_ref - p0)):
        assert rel_to_max(a, b) <= 3e-2, ("update", name)
