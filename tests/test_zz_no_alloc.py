"""The allocation-free softmax cross-entropy entry point.

softmax_xent_fwd_bwd_noalloc serves callers that cannot allocate device
memory (a host framework that owns the device heap, an allocator callback, a
runtime that forbids allocation after start-up): it keeps its scratch in a
fixed device array inside the library instead of a caller workspace.  These
tests call it through the C ABI twice in a row, on different inputs, on each
of the loss kernel's paths (one row per thread for small heads, one block for
small batches, per-block partial sums in the scratch for large batches), and
check each result bit for bit against softmax_xent_fwd_bwd with a caller
workspace (the same kernels in the same order), against the oracle's softmax
cross entropy, and that the calls leave the device's free memory unchanged.
The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import mlp_step_gb300 as M
from mlp_step_gb300 import synth

pytestmark = pytest.mark.gpu


def _inputs(B, C, seed):
    Z = torch.from_numpy(synth.normal_f32((B, C), synth.STREAM_GENERIC + seed, std=3.0)).cuda()
    y = torch.from_numpy(synth.labels(B, C, seed=seed)).cuda()
    return Z, y


def _noalloc(Z, y, loss, dl, am):
    B, C = Z.shape
    return M.load().softmax_xent_fwd_bwd_noalloc(
        ctypes.c_void_p(Z.data_ptr()), C, ctypes.c_void_p(y.data_ptr()), B, C,
        ctypes.c_void_p(loss.data_ptr()), ctypes.c_void_p(dl.data_ptr()), M.MLP_DTYPE_F32,
        dl.shape[1], ctypes.c_void_p(am.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _outputs(B, ld):
    return (torch.full((4,), float("nan"), device="cuda"),
            torch.full((B, ld), float("nan"), device="cuda"),
            torch.full((B,), -1, dtype=torch.int32, device="cuda"))


# (batch, classes): one row per thread (C <= 32, B <= 512); one block
# (B <= 256); per-block partial sums in the scratch array
CASES = [(300, 10), (200, 1000), (16421, 1000)]


@pytest.mark.parametrize("B,C", CASES)
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(B, C):
    M.load()
    ld = (C + 7) // 8 * 8
    # the first call on the device does the scratch set-up; the calls after it
    # allocate nothing
    Z0, y0 = _inputs(B, C, 0)
    assert _noalloc(Z0, y0, *_outputs(B, ld)) == M.MLP_OK
    for seed in (1, 2):
        Z, y = _inputs(B, C + 0, seed)
        ref = _outputs(B, ld)
        ws = torch.empty(max(M.softmax_xent_workspace_bytes(B, C), 16), dtype=torch.uint8,
                         device="cuda")
        M.softmax_xent_fwd_bwd(Z, y, ref[0], dlogits=ref[1], argmax_out=ref[2], workspace=ws)
        got = _outputs(B, ld)
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        used0 = torch.cuda.memory_allocated()
        assert _noalloc(Z, y, *got) == M.MLP_OK
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        assert torch.cuda.memory_allocated() == used0
        # the same kernels in the same order: identical results
        assert torch.equal(got[0][:1], ref[0][:1])
        assert torch.equal(got[1], ref[1])
        assert torch.equal(got[2], ref[2])
        # and the oracle's definition (fp64): mean loss, dZ, argmax
        L, _, dZ, am = oracle.softmax_xent(Z.double().cpu().numpy(), y.cpu().numpy())
        assert abs(got[0][0].item() - L) <= 1e-5 * abs(L)
        d = got[1].cpu().numpy()[:, :C]
        assert np.all(np.abs(d - dZ) <= 1e-6 / B + 1e-5 * np.abs(dZ))
        assert np.all(got[1].cpu().numpy()[:, C:] == 0.0)
        assert np.array_equal(got[2].cpu().numpy(), am)
    assert M.get_device_status() == M.MLP_OK


def test_noalloc_rejects_batches_above_its_scratch():
    lib = M.load()
    top = lib.softmax_xent_noalloc_max_batch()
    assert top == 524288   # 65,536 partials of 8 rows each
    fake = ctypes.c_void_p(0x10000)
    st = lib.softmax_xent_fwd_bwd_noalloc(fake, 10, fake, top + 1, 10, fake, None, 0, 10, None,
                                          None)
    assert st == M.MLP_ERR_UNSUPPORTED_SHAPE
