"""The allocation-free softmax cross-entropy entry point.

softmax_xent_fwd_bwd_noalloc serves callers that cannot allocate device
memory (a host framework that owns the device heap, an allocator callback, a
runtime that forbids allocation after start-up): it keeps its scratch in a
fixed device array inside the library instead of a caller workspace.  This
test calls it through the C ABI twice in a row, on different inputs, and
checks each result against softmax_xent_fwd_bwd with a caller workspace.  The
file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import mlp_step_gb300 as M
from mlp_step_gb300 import synth

pytestmark = pytest.mark.gpu


def _run_both(B, C, seed):
    Z = torch.from_numpy(synth.normal_f32((B, C), synth.STREAM_GENERIC + seed, std=3.0)).cuda()
    y = torch.from_numpy(synth.labels(B, C, seed=seed)).cuda()
    ld = (C + 7) // 8 * 8
    outs = []
    for noalloc in (False, True):
        loss = torch.full((4,), float("nan"), device="cuda")
        dl = torch.full((B, ld), float("nan"), device="cuda")
        am = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        if noalloc:
            st = M.load().softmax_xent_fwd_bwd_noalloc(
                ctypes.c_void_p(Z.data_ptr()), C, ctypes.c_void_p(y.data_ptr()), B, C,
                ctypes.c_void_p(loss.data_ptr()), ctypes.c_void_p(dl.data_ptr()),
                M.MLP_DTYPE_F32, ld, ctypes.c_void_p(am.data_ptr()),
                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
            assert st == M.MLP_OK, M.status_string(st)
        else:
            ws = torch.empty(max(M.softmax_xent_workspace_bytes(B, C), 16), dtype=torch.uint8,
                             device="cuda")
            M.softmax_xent_fwd_bwd(Z, y, loss, dlogits=dl, argmax_out=am, workspace=ws)
        torch.cuda.synchronize()
        outs.append((loss[0].item(), dl.cpu().numpy(), am.cpu().numpy()))
    return outs


def test_noalloc_matches_workspace_entry_point_twice():
    M.load()
    # large enough that the mean goes through the scratch partials
    for seed in (1, 2):
        (l_ref, d_ref, a_ref), (l, d, a) = _run_both(16384 + 37 * seed, 1000, seed)
        assert abs(l - l_ref) <= 2e-6 * max(1.0, abs(l_ref))
        assert np.all(np.abs(d - d_ref) <= 1e-7 + 1e-5 * np.abs(d_ref))
        assert np.array_equal(a, a_ref)
    assert M.get_device_status() == M.MLP_OK


def test_noalloc_rejects_batches_above_its_scratch():
    lib = M.load()
    assert lib.softmax_xent_noalloc_max_batch() == 524288
    fake = ctypes.c_void_p(0x10000)
    st = lib.softmax_xent_fwd_bwd_noalloc(fake, 10, fake, 524289, 10, fake, None, 0, 10, None,
                                          None)
    assert st == M.MLP_ERR_UNSUPPORTED_SHAPE
