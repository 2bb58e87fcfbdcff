"""Parity of the fused attention preprocessing ("Full-Depth MLP Megakernel +
Fused Attention Preprocessing", "What Worked" and "What Didn't Work": RMSNorm
-> QKV projection -> QK norm -> partial RoPE -> q gain) with the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import mlp_step_gb300 as M
from mlp_step_gb300 import synth
from helpers import bf16_values, to_dev, rel_to_max, assert_elementwise

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    M.load()
    yield
    assert M.get_device_status() == M.MLP_OK


def _inputs(T, d, n_q, n_kv, seed=0):
    N = (n_q + 2 * n_kv) * 64
    x = synth.normal_f32((T, d), synth.STREAM_GENERIC + seed)
    W = synth.normal_f32((d, N), synth.STREAM_GENERIC + seed + 1, std=d ** -0.5)
    gain = synth.uniform_f32((n_q,), synth.STREAM_GENERIC + seed + 2, lo=0.5, hi=1.5)
    return x, W, gain


def _run(x, W, gain, n_q, n_kv, R, seq_len, eps=1e-6):
    T, d = x.shape
    N = W.shape[1]
    out = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    rstd = torch.empty(T, device="cuda")
    M.mlp_attn_prep_fwd(to_dev(x, torch.bfloat16), to_dev(W, torch.bfloat16), to_dev(gain), out,
                        rstd, n_q, n_kv, R, seq_len, eps=eps)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), rstd.cpu().numpy()


def _check(got, ref, n_q, n_kv):
    assert np.all(np.isfinite(got)), "unwritten outputs"
    hq, hk = n_q * 64, (n_q + n_kv) * 64
    for name, a, b in (("q", 0, hq), ("k", hq, hk), ("v", hk, got.shape[1])):
        # bf16 output (2^-9 relative) of fp32-accumulated values
        assert rel_to_max(got[:, a:b], ref[:, a:b]) <= 8e-3, name
        assert_elementwise(got[:, a:b], ref[:, a:b], 8e-3, 8e-3 * np.abs(ref[:, a:b]).max(), name)


@pytest.mark.parametrize("T,d,n_q,n_kv,R,seq_len", [(1000, 512, 8, 4, 32, 128),
                                                    (300, 136, 2, 1, 16, 7),
                                                    (513, 512, 4, 4, 64, 1024),
                                                    (1, 64, 1, 1, 32, 1),
                                                    (300, 1024, 2, 1, 32, 64)])
def test_attn_prep_matches_oracle(T, d, n_q, n_kv, R, seq_len):
    x, W, gain = _inputs(T, d, n_q, n_kv)
    got, rstd = _run(x, W, gain, n_q, n_kv, R, seq_len)
    ref = oracle.attn_prep(bf16_values(x), bf16_values(W), gain.astype(np.float64), n_q, n_kv,
                           64, R, seq_len)
    _check(got, ref, n_q, n_kv)
    xb = bf16_values(x)
    assert np.allclose(rstd, 1.0 / np.sqrt((xb * xb).mean(1) + 1e-6), rtol=1e-5)


def test_attn_prep_full_size_sampled_rows():
    """The bench workload's shape (65,536 tokens of 512, 8 query and 4 key /
    value heads of 64, RoPE on 32 dims, sequences of 1,024): sampled rows,
    including both ends of sequences and the last token."""
    T, d, n_q, n_kv, R, L = 65536, 512, 8, 4, 32, 1024
    x, W, gain = _inputs(T, d, n_q, n_kv, seed=3)
    got, _ = _run(x, W, gain, n_q, n_kv, R, L)
    rows = np.unique(np.concatenate([[0, 1, L - 1, L, 2 * L + 5, T - 1],
                                     synth.randint(11, synth.STREAM_GENERIC, 40, T)]))
    ref = oracle.attn_prep_rows(bf16_values(x).astype(np.float32),
                                bf16_values(W).astype(np.float32), gain, rows, n_q, n_kv, 64, R, L)
    _check(got[rows], ref, n_q, n_kv)


def test_attn_prep_weights_reloaded_across_tile_columns():
    """K up to 512 keeps a CTA pair's 256 weight columns resident while it
    walks a run of token tiles down one column; with three columns (N = 640,
    the last one ragged) over 79 token tiles, some runs cross into the next
    column and load its weights mid-run.  Two rows of every 256-token tile,
    one from each CTA of the pair, against the oracle."""
    T, d, n_q, n_kv, R, L = 20000, 512, 6, 2, 32, 1000
    x, W, gain = _inputs(T, d, n_q, n_kv, seed=5)
    got, _ = _run(x, W, gain, n_q, n_kv, R, L)
    tiles = np.arange((T + 255) // 256)
    rows = np.unique(np.minimum(np.concatenate([tiles * 256 + (tiles * 37) % 128,
                                                tiles * 256 + 128 + (tiles * 53) % 128,
                                                [T - 1]]), T - 1))
    ref = oracle.attn_prep_rows(bf16_values(x).astype(np.float32),
                                bf16_values(W).astype(np.float32), gain, rows, n_q, n_kv, 64, R, L)
    _check(got[rows], ref, n_q, n_kv)
