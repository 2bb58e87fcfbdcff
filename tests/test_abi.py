"""Host-side checks of the C ABI: the library loads without a GPU, exports
every function include/mlp_step.h declares, and rejects bad arguments before
enqueueing anything (none of these calls launches a kernel)."""
import ctypes
import os
import re

import pytest

import mlp_step_gb300 as M
from mlp_step_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return M.load()


def _declared_functions():
    txt = open(os.path.join(ROOT, "include", "mlp_step.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", txt)
    skip = {"if", "sizeof", "defined"}
    return sorted(set(n for n in names if n not in skip))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 25
    for n in names:
        assert hasattr(lib, n), n
        assert n in M.SIGNATURES, n


def test_param_count_and_offsets(lib):
    assert M.mlp_param_count([784, 256, 10]) == 203530
    assert M.mlp_param_count([1024, 8192, 8192, 1000]) == 83706856
    assert M.mlp_param_offset([784, 256, 10], 0, 0) == 0
    assert M.mlp_param_offset([784, 256, 10], 0, 1) == 200704
    assert M.mlp_param_offset([784, 256, 10], 1, 0) == 200960
    assert M.mlp_param_offset([784, 256, 10], 1, 1) == 203520
    assert M.mlp_param_offset([784, 256, 10], 2, 0) == ctypes.c_size_t(-1).value
    # W2 [256][10] is padded to 16 columns in the bf16 shadow
    assert M.mlp_shadow_elems([784, 256, 10]) == 784 * 256 + 256 * 16
    assert M.mlp_param_count([784]) == 0


def test_status_strings(lib):
    for s in range(7):
        assert M.status_string(s)
    assert M.status_string(99) == "unknown status"


def test_create_rejects_bad_arguments(lib):
    d = (ctypes.c_int * 3)(784, 256, 10)
    h = ctypes.c_void_p()
    fake = ctypes.c_void_p(0x10000)
    # null buffers
    assert lib.mlp_create(d, 3, 1, 1, 128, None, None, None, None, None, 0, ctypes.byref(h)) == 1
    # workspace too small
    assert lib.mlp_create(d, 3, 1, 0, 128, fake, fake, fake, None, fake, 16, ctypes.byref(h)) == 1
    # misaligned parameter pointer
    need = M.mlp_workspace_bytes([784, 256, 10], 128, 0)
    bad = ctypes.c_void_p(0x10004)
    assert lib.mlp_create(d, 3, 1, 0, 128, bad, fake, fake, None, fake, need, ctypes.byref(h)) == 2
    # the 16-bit tensor-core precisions need the weight shadow
    need16 = M.mlp_workspace_bytes([784, 256, 10], 128, M.MLP_PREC_FP16)
    assert need16 == M.mlp_workspace_bytes([784, 256, 10], 128, M.MLP_PREC_BF16) > 0
    for prec in (M.MLP_PREC_BF16, M.MLP_PREC_FP16):
        assert lib.mlp_create(d, 3, 1, prec, 128, fake, fake, fake, None, fake, need16,
                              ctypes.byref(h)) == 1
    # unknown precision / activation
    assert lib.mlp_create(d, 3, 1, 7, 128, fake, fake, fake, None, fake, need, ctypes.byref(h)) == 1
    assert lib.mlp_create(d, 3, 9, 0, 128, fake, fake, fake, None, fake, need, ctypes.byref(h)) == 1


def test_gemm_rejects_bad_arguments(lib):
    fake = ctypes.c_void_p(0x10000)
    # ldc < N
    assert lib.mlp_gemm(4, 8, 8, fake, 8, 0, fake, 8, 0, 1, None, 0, None, 0, fake, 4, 0, None) == 1
    # bf16 row pitch not 16-byte aligned (lda = 10 elements = 20 B)
    assert lib.mlp_gemm(4, 8, 10, fake, 10, 0, fake, 8, 0, 1, None, 0, None, 0, fake, 8, 0,
                        None) == 2
    # unknown activation
    assert lib.mlp_gemm(4, 8, 8, fake, 8, 0, fake, 8, 0, 1, None, 5, None, 0, fake, 8, 0, None) == 1
    # empty problem: OK, nothing launched
    assert lib.mlp_gemm(0, 8, 8, None, 8, 0, None, 8, 0, 1, None, 0, None, 0, None, 8, 0, None) == 0
    # 16-bit outputs take the operands' 16-bit type: fp16 in -> bf16 out and
    # bf16 in -> fp16 out are rejected; an fp16 row pitch must be 16-byte aligned
    F16, BF16 = M.MLP_DTYPE_F16, M.MLP_DTYPE_BF16
    assert lib.mlp_gemm(4, 8, 8, fake, 8, 0, fake, 8, 0, F16, None, 0, None, 0, fake, 8, BF16,
                        None) == 1
    assert lib.mlp_gemm(4, 8, 8, fake, 8, 0, fake, 8, 0, BF16, None, 0, None, 0, fake, 8, F16,
                        None) == 1
    assert lib.mlp_gemm(4, 8, 10, fake, 10, 0, fake, 8, 0, F16, None, 0, None, 0, fake, 8, F16,
                        None) == 2


def test_other_entry_points_reject_bad_arguments(lib):
    fake = ctypes.c_void_p(0x10000)
    assert lib.softmax_xent_fwd_bwd(None, 10, fake, 128, 10, None, None, 0, 10, None, None, 0,
                                    None) == 1
    assert lib.softmax_xent_fwd_bwd(fake, 10, fake, 0, 10, None, None, 0, 10, None, None, 0,
                                    None) == 0
    assert lib.sgd_momentum_step(None, None, None, None, 10, 0.1, 0.9, None) == 1
    assert lib.sgd_momentum_step(None, None, None, None, 0, 0.1, 0.9, None) == 0
    assert lib.sgd_momentum_step(ctypes.c_void_p(0x10004), fake, fake, None, 10, 0.1, 0.9,
                                 None) == 2
    assert lib.mlp_colsum(fake, 7, 4, 4, 4, fake, None, 0, None) == 1
    assert lib.mse_loss_fwd_bwd(fake, fake, 100, fake, fake, None, 0, None) == 1
    assert lib.mlp_selftest_wait_timeout(0, None) == 1


def test_block_and_stack_entry_points_check_shapes_and_pointers(lib):
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)  # 8-byte aligned only
    f = ctypes.c_float
    # forward: negative T, unsupported width / hidden size, negative eps
    assert lib.mlp_block_fwd(fake, fake, fake, -1, 512, 1536, f(1e-6), f(0.5), fake, fake,
                             None) == 1
    assert lib.mlp_block_fwd(fake, fake, fake, 8, 256, 1536, f(1e-6), f(0.5), fake, fake,
                             None) == 3
    assert lib.mlp_block_fwd(fake, fake, fake, 8, 512, 1000, f(1e-6), f(0.5), fake, fake,
                             None) == 3
    assert lib.mlp_block_fwd(fake, fake, fake, 8, 512, 1536, f(-1.0), f(0.5), fake, fake,
                             None) == 1
    # empty: nothing to do; null pointers are fine then
    assert lib.mlp_block_fwd(None, None, None, 0, 512, 1536, f(1e-6), f(0.5), None, None,
                             None) == 0
    assert lib.mlp_block_fwd(None, fake, fake, 8, 512, 1536, f(1e-6), f(0.5), fake, fake,
                             None) == 1
    assert lib.mlp_block_fwd(odd, fake, fake, 8, 512, 1536, f(1e-6), f(0.5), fake, fake,
                             None) == 2
    # backward: workspace too small, empty, misaligned
    need = M.mlp_block_workspace_bytes(8, 512, 1536)
    assert need > 0 and M.mlp_block_workspace_bytes(8, 512, 1000) == 0
    args = [fake, fake, fake, fake, fake, 8, 512, 1536, f(1e-6), f(0.5), fake, fake, fake, fake]
    assert lib.mlp_block_bwd(*args, need - 1, None) == 1
    assert lib.mlp_block_bwd(*args[:5], 0, *args[6:], 0, None) == 0
    assert lib.mlp_block_bwd(odd, *args[1:], need, None) == 2
    # stack: no blocks, empty, workspace too small
    P = M.mlp_stack_param_count(2, 512, 1536)
    assert P == 2 * 2 * 512 * 1536
    ws = M.mlp_stack_workspace_bytes(2, 8, 512, 1536)
    st = [fake, fake, fake, fake, fake, fake, f(0.02), f(0.95), fake, fake]
    assert lib.mlp_stack_train_step(0, 8, 512, 1536, f(1e-6), f(0.5), *st, ws, None) == 1
    assert lib.mlp_stack_train_step(2, 0, 512, 1536, f(1e-6), f(0.5), *st, ws, None) == 0
    assert lib.mlp_stack_train_step(2, 8, 512, 1536, f(1e-6), f(0.5), *st, ws - 1, None) == 1
    assert lib.mlp_stack_train_step(2, 8, 512, 1000, f(1e-6), f(0.5), *st, ws, None) == 3


def test_loss_and_update_entry_points_check_arguments(lib):
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10004)
    f = ctypes.c_float
    # softmax cross entropy: no classes, leading dimensions below the width,
    # unknown dZ type
    assert lib.softmax_xent_fwd_bwd(fake, 10, fake, 4, 0, None, None, 0, 10, None, None, 0,
                                    None) == 1
    assert lib.softmax_xent_fwd_bwd(fake, 8, fake, 4, 10, None, None, 0, 10, None, None, 0,
                                    None) == 1
    assert lib.softmax_xent_fwd_bwd(fake, 10, fake, 4, 10, None, fake, 0, 8, None, None, 0,
                                    None) == 1
    assert lib.softmax_xent_fwd_bwd(fake, 10, fake, 4, 10, None, fake, 9, 16, None, None, 0,
                                    None) == 1
    # MSE: empty, misaligned input
    assert lib.mse_loss_fwd_bwd(None, None, 0, None, None, None, 0, None) == 0
    ws = M.mse_workspace_bytes(100)
    assert lib.mse_loss_fwd_bwd(odd, fake, 100, fake, fake, fake, ws, None) == 2
    # column sums: negative rows, nothing to sum, ld below the width
    assert lib.mlp_colsum(fake, 0, -1, 4, 4, fake, None, 0, None) == 1
    assert lib.mlp_colsum(None, 0, 4, 0, 4, None, None, 0, None) == 0
    assert lib.mlp_colsum(fake, 0, 4, 8, 4, fake, None, 0, None) == 1
    # GEMM: negative sizes, empty output, unknown activation
    g = [fake, 8, 0, fake, 8, 0, 0, None, 0, None, 0, fake, 8, 0, None]
    assert lib.mlp_gemm(-1, 8, 8, *g) == 1
    assert lib.mlp_gemm(0, 8, 8, *g) == 0
    assert lib.mlp_gemm(8, 0, 8, *g) == 0
    assert lib.mlp_gemm(8, 8, 8, fake, 8, 0, fake, 8, 0, 0, None, 5, None, 0, fake, 8, 0,
                        None) == 1
    # training entry points without a handle
    assert lib.mlp_train_step(None, fake, 2, fake, 128, f(0.1), f(0.9), None, None, None) == 1
    assert lib.mlp_train_epoch(None, fake, 2, fake, 256, 128, f(0.1), f(0.9), None, None,
                               None) == 1
    assert lib.mlp_forward(None, fake, 2, 128, fake, None) == 1


def test_attn_prep_entry_point_checks_arguments(lib):
    fake = ctypes.c_void_p(0x10000)
    f = ctypes.c_float
    call = lambda T, d, nq, nkv, hd, R, L, x=fake, out=fake: lib.mlp_attn_prep_fwd(
        x, fake, fake, T, d, nq, nkv, hd, R, L, f(1e-6), f(10000.0), out, fake, None)
    assert call(0, 512, 8, 4, 64, 32, 1024) == 0                     # empty: nothing launched
    assert call(-1, 512, 8, 4, 64, 32, 1024) == 1
    assert call(16, 512, 0, 4, 64, 32, 1024) == 1                    # no query heads
    assert call(16, 512, 8, 4, 128, 32, 1024) == 3                   # head_dim must be 64
    assert call(16, 512, 8, 4, 64, 24, 1024) == 3                    # rope dims 16 / 32 / 64
    assert call(16, 500, 8, 4, 64, 32, 1024) == 3                    # rows of 8 bf16
    assert call(16, 512, 8, 4, 64, 32, 1024, x=None) == 1
    assert call(16, 512, 8, 4, 64, 32, 1024, out=ctypes.c_void_p(0x10008)) == 2


def test_reduction_order_switch(lib):
    assert M.get_reduction_order() == M.MLP_ORDER_FAST
    assert lib.mlp_set_reduction_order(7) == 1          # unknown order: rejected, unchanged
    assert M.get_reduction_order() == M.MLP_ORDER_FAST
    M.set_reduction_order(M.MLP_ORDER_LINEAR)
    try:
        assert M.get_reduction_order() == M.MLP_ORDER_LINEAR
    finally:
        M.set_reduction_order(M.MLP_ORDER_FAST)
    assert M.get_reduction_order() == M.MLP_ORDER_FAST


def test_byte_scaling_by_reciprocal_rounds_like_division():
    """The cast of image bytes to a 16-bit operand multiplies by fp32(1/255)
    instead of dividing by 255: for every byte the product rounds to the same
    bf16 and fp16 value as the IEEE fp32 quotient byte / 255 (the value the
    oracle and the fp32 path use), so the shortcut changes no result."""
    import numpy as np
    import torch
    b = np.arange(256, dtype=np.float32)
    q = b / np.float32(255)
    m = b * (np.float32(1) / np.float32(255))
    for dt in (torch.bfloat16, torch.float16):
        assert torch.equal(torch.from_numpy(q).to(dt), torch.from_numpy(m).to(dt)), dt
