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
