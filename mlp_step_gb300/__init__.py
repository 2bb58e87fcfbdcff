"""GB300-native MLP training step: CUDA kernels for sm_103a behind a C ABI.

This module is the thin Python binding of ``libmlp_step.so`` (declared in
``include/mlp_step.h``).  It only marshals arguments: tensors become device
pointers, the current torch CUDA stream becomes the ``cudaStream_t``, and a
non-zero status becomes :class:`MlpError`.  Every step of the computation runs
in the library's kernels; if the library is missing, calls raise instead of
falling back to anything else.

PyTorch supplies device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "MlpError", "load", "lib_path",
    "MLP_ACT_NONE", "MLP_ACT_RELU", "MLP_ACT_LEAKY_RELU_SQ",
    "MLP_PREC_FP32", "MLP_PREC_BF16", "MLP_PREC_FP16", "MLP_DTYPE_F32", "MLP_DTYPE_BF16",
    "MLP_DTYPE_U8", "MLP_DTYPE_F16", "MLP_ORDER_FAST", "MLP_ORDER_LINEAR",
]

MLP_OK = 0
MLP_ERR_INVALID_ARG = 1
MLP_ERR_MISALIGNED = 2
MLP_ERR_UNSUPPORTED_SHAPE = 3
MLP_ERR_CUDA = 4
MLP_ERR_DEVICE_TIMEOUT = 5
MLP_ERR_NUMERIC = 6

MLP_ACT_NONE = 0
MLP_ACT_RELU = 1
MLP_ACT_LEAKY_RELU_SQ = 2
MLP_PREC_FP32 = 0
MLP_PREC_BF16 = 1
MLP_PREC_FP16 = 2
MLP_DTYPE_F32 = 0
MLP_DTYPE_BF16 = 1
MLP_DTYPE_U8 = 2
MLP_DTYPE_F16 = 3
MLP_ORDER_FAST = 0
MLP_ORDER_LINEAR = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libmlp_step.so")
_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t
_ll = ctypes.c_longlong

# name -> (restype, argtypes); the signatures of include/mlp_step.h
SIGNATURES = {
    "mlp_status_string": (ctypes.c_char_p, [_i]),
    "mlp_get_device_status": (_i, [_vp]),
    "mlp_set_wait_limit_ns": (None, [_ll]),
    "mlp_set_reduction_order": (_i, [_i]),
    "mlp_attn_prep_fwd": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, ctypes.c_float,
                               ctypes.c_float, _vp, _vp, _vp]),
    "mlp_get_reduction_order": (_i, []),
    "mlp_selftest_wait_timeout": (_i, [_ll, _vp]),
    "mlp_launch_count": (ctypes.c_ulonglong, []),
    "mlp_timing_enable": (_i, [_i]),
    "mlp_timing_report": (_sz, [ctypes.c_char_p, _sz]),
    "mlp_param_count": (_sz, [_vp, _i]),
    "mlp_param_offset": (_sz, [_vp, _i, _i, _i]),
    "mlp_shadow_elems": (_sz, [_vp, _i]),
    "mlp_workspace_bytes": (_sz, [_vp, _i, _i, _i]),
    "mlp_create": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _sz, ctypes.POINTER(_vp)]),
    "mlp_destroy": (None, [_vp]),
    "mlp_refresh_shadow": (_i, [_vp, _vp]),
    "mlp_forward": (_i, [_vp, _vp, _i, _i, _vp, _vp]),
    "mlp_backward": (_i, [_vp, _vp, _i, _i, _vp, _vp]),
    "mlp_sgd_step": (_i, [_vp, _f, _f, _vp]),
    "mlp_train_step": (_i, [_vp, _vp, _i, _vp, _i, _f, _f, _vp, _vp, _vp]),
    "mlp_train_epoch": (_i, [_vp, _vp, _i, _vp, _i, _i, _f, _f, _vp, _vp, _vp]),
    "softmax_xent_workspace_bytes": (_sz, [_i, _i]),
    "softmax_xent_fwd_bwd": (_i, [_vp, _i, _vp, _i, _i, _vp, _vp, _i, _i, _vp, _vp, _sz, _vp]),
    "softmax_xent_noalloc_max_batch": (_i, []),
    "softmax_xent_fwd_bwd_noalloc": (_i, [_vp, _i, _vp, _i, _i, _vp, _vp, _i, _i, _vp, _vp]),
    "sgd_momentum_step": (_i, [_vp, _vp, _vp, _vp, _sz, _f, _f, _vp]),
    "mlp_gemm": (_i, [_i, _i, _i, _vp, _i, _i, _vp, _i, _i, _i, _vp, _i, _vp, _i, _vp, _i, _i,
                      _vp]),
    "mlp_colsum_workspace_bytes": (_sz, [_i, _i]),
    "mlp_colsum": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "mlp_block_workspace_bytes": (_sz, [_i, _i, _i]),
    "mlp_block_fwd": (_i, [_vp, _vp, _vp, _i, _i, _i, _f, _f, _vp, _vp, _vp]),
    "mlp_block_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _f, _f, _vp, _vp, _vp, _vp, _sz,
                           _vp]),
    "mse_workspace_bytes": (_sz, [_sz]),
    "mse_loss_fwd_bwd": (_i, [_vp, _vp, _sz, _vp, _vp, _vp, _sz, _vp]),
    "mlp_stack_param_count": (_sz, [_i, _i, _i]),
    "mlp_stack_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "mlp_stack_train_step": (_i, [_i, _i, _i, _i, _f, _f, _vp, _vp, _vp, _vp, _vp, _vp, _f, _f,
                                  _vp, _vp, _sz, _vp]),
}


class MlpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = load().mlp_status_string(status).decode() if _lib is not None else str(status)
        super().__init__("%s: %s (status %d)" % (where, msg, status))


def load():
    """Loads libmlp_step.so (built by ``mlp_step_gb300.build``); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(lib_path):
            raise ImportError("libmlp_step.so is not built; run mlp_step_gb300.build.build()")
        lib = ctypes.CDLL(lib_path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


# ------------------------------------------------------------------ helpers

def _ptr(t):
    """Device address of a tensor the library reads as row-major rows: the
    last dimension must be unit-stride (rows may be padded, their pitch is
    passed as the leading dimension), and tensors of more than two
    dimensions must be contiguous."""
    if t is None:
        return None
    if t.dim() >= 1 and t.numel() > 1 and t.stride(-1) != 1:
        raise ValueError("the library reads row-major rows: last dimension must have stride 1 "
                         "(got strides %s)" % (tuple(t.stride()),))
    if t.dim() > 2 and not t.is_contiguous():
        raise ValueError("tensors of more than two dimensions must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, where):
    if status != MLP_OK:
        raise MlpError(status, where)


def _dims(dims):
    return (ctypes.c_int * len(dims))(*dims), len(dims)


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return MLP_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return MLP_DTYPE_BF16
    if t.dtype == torch.uint8:
        return MLP_DTYPE_U8
    if t.dtype == torch.float16:
        return MLP_DTYPE_F16
    raise TypeError("unsupported dtype %s" % t.dtype)


# ------------------------------------------------------------------ status

def status_string(s: int) -> str:
    return load().mlp_status_string(s).decode()


def get_device_status(stream=None) -> int:
    return load().mlp_get_device_status(_stream(stream))


def set_wait_limit_ns(ns: int) -> None:
    load().mlp_set_wait_limit_ns(int(ns))


def set_reduction_order(order: int) -> None:
    """MLP_ORDER_FAST or MLP_ORDER_LINEAR (see mlp_step.h)."""
    _check(load().mlp_set_reduction_order(int(order)), "mlp_set_reduction_order")


def get_reduction_order() -> int:
    return load().mlp_get_reduction_order()


def selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(load().mlp_selftest_wait_timeout(int(limit_ns), _stream(stream)),
           "mlp_selftest_wait_timeout")


def launch_count() -> int:
    """Kernels enqueued (or captured) by the library since it was loaded."""
    return load().mlp_launch_count()


def timing_enable(on: bool) -> None:
    load().mlp_timing_enable(1 if on else 0)


def timing_report() -> dict:
    """{"kernel[shape]": (launches, total_ms)} for launches since timing_enable(True)."""
    import json
    L = load()
    need = L.mlp_timing_report(None, 0)
    buf = ctypes.create_string_buffer(need + 16)
    L.mlp_timing_report(buf, len(buf))
    return {k: (v[0], v[1]) for k, v in json.loads(buf.value.decode()).items()}


# ------------------------------------------------------------------ MLP

def mlp_param_count(dims) -> int:
    d, n = _dims(dims)
    return load().mlp_param_count(d, n)


def mlp_param_offset(dims, layer: int, which: int) -> int:
    d, n = _dims(dims)
    return load().mlp_param_offset(d, n, layer, which)


def mlp_shadow_elems(dims) -> int:
    d, n = _dims(dims)
    return load().mlp_shadow_elems(d, n)


def mlp_workspace_bytes(dims, max_batch: int, prec: int) -> int:
    d, n = _dims(dims)
    return load().mlp_workspace_bytes(d, n, max_batch, prec)


class MLP:
    """Owner of the device buffers of one MLP (flat params, velocity, grads,
    the 16-bit weight shadow of the tensor-core precisions, workspace) and of
    the library handle over them."""

    def __init__(self, dims, prec=MLP_PREC_BF16, max_batch=128, params=None,
                 hidden_act=MLP_ACT_RELU, device="cuda"):
        import torch
        self.dims = list(dims)
        self.prec = prec
        self.max_batch = max_batch
        n = mlp_param_count(self.dims)
        self.params = torch.zeros(n, dtype=torch.float32, device=device)
        if params is not None:
            self.params.copy_(torch.as_tensor(params, dtype=torch.float32))
        self.velocity = torch.zeros_like(self.params)
        self.grads = torch.zeros_like(self.params)
        self.shadow = None
        if prec in (MLP_PREC_BF16, MLP_PREC_FP16):
            self.shadow = torch.zeros(mlp_shadow_elems(self.dims),
                                      dtype=torch.bfloat16 if prec == MLP_PREC_BF16
                                      else torch.float16, device=device)
        wsb = mlp_workspace_bytes(self.dims, max_batch, prec)
        self.workspace = torch.empty(wsb, dtype=torch.uint8, device=device)
        d, nd = _dims(self.dims)
        h = ctypes.c_void_p()
        _check(load().mlp_create(d, nd, hidden_act, prec, max_batch, _ptr(self.params),
                                 _ptr(self.velocity), _ptr(self.grads), _ptr(self.shadow),
                                 _ptr(self.workspace), wsb, ctypes.byref(h)), "mlp_create")
        self.handle = h
        self.refresh_shadow()

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.mlp_destroy(self.handle)
            self.handle = None

    def refresh_shadow(self, stream=None):
        _check(load().mlp_refresh_shadow(self.handle, _stream(stream)), "mlp_refresh_shadow")

    def forward(self, x, logits, stream=None):
        _check(load().mlp_forward(self.handle, _ptr(x), _dtype_code(x), x.shape[0], _ptr(logits),
                                  _stream(stream)), "mlp_forward")

    def backward(self, dlogits, batch, dx=None, stream=None):
        _check(load().mlp_backward(self.handle, _ptr(dlogits), dlogits.shape[1], batch, _ptr(dx),
                                   _stream(stream)), "mlp_backward")

    def sgd_step(self, lr, momentum, stream=None):
        _check(load().mlp_sgd_step(self.handle, lr, momentum, _stream(stream)), "mlp_sgd_step")

    def train_step(self, x, labels, lr, momentum, loss_out=None, argmax_out=None, batch=None,
                   stream=None):
        b = x.shape[0] if batch is None else batch
        _check(load().mlp_train_step(self.handle, _ptr(x), _dtype_code(x), _ptr(labels), b, lr,
                                     momentum, _ptr(loss_out), _ptr(argmax_out),
                                     _stream(stream)), "mlp_train_step")

    def train_epoch(self, x, labels, lr, momentum, batch, losses_out=None, argmax_out=None,
                    n_samples=None, stream=None):
        """Training steps over x / labels in order, `batch` rows at a time (the
        last step takes the remainder); losses_out: fp32[n_steps]."""
        n = x.shape[0] if n_samples is None else n_samples
        _check(load().mlp_train_epoch(self.handle, _ptr(x), _dtype_code(x), _ptr(labels), n,
                                      batch, lr, momentum, _ptr(losses_out), _ptr(argmax_out),
                                      _stream(stream)), "mlp_train_epoch")


# ------------------------------------------------------------------ single kernels

def softmax_xent_workspace_bytes(batch: int, classes: int) -> int:
    return load().softmax_xent_workspace_bytes(batch, classes)


def softmax_xent_fwd_bwd(logits, labels, loss_out, dlogits=None, argmax_out=None,
                         workspace=None, classes=None, stream=None):
    B = logits.shape[0]
    C = logits.shape[1] if classes is None else classes
    dl_dtype = _dtype_code(dlogits) if dlogits is not None else MLP_DTYPE_F32
    ldd = dlogits.shape[1] if dlogits is not None else C
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().softmax_xent_fwd_bwd(_ptr(logits), logits.stride(0), _ptr(labels), B, C,
                                       _ptr(loss_out), _ptr(dlogits), dl_dtype, ldd,
                                       _ptr(argmax_out), _ptr(workspace), wsb, _stream(stream)),
           "softmax_xent_fwd_bwd")


def softmax_xent_fwd_bwd_noalloc(logits, labels, loss_out, dlogits=None, argmax_out=None,
                                 classes=None, stream=None):
    """softmax_xent_fwd_bwd with the library's fixed device scratch (no workspace)."""
    B = logits.shape[0]
    C = logits.shape[1] if classes is None else classes
    dl_dtype = _dtype_code(dlogits) if dlogits is not None else MLP_DTYPE_F32
    ldd = dlogits.shape[1] if dlogits is not None else C
    _check(load().softmax_xent_fwd_bwd_noalloc(_ptr(logits), logits.stride(0), _ptr(labels), B,
                                               C, _ptr(loss_out), _ptr(dlogits), dl_dtype, ldd,
                                               _ptr(argmax_out), _stream(stream)),
           "softmax_xent_fwd_bwd_noalloc")


def sgd_momentum_step(w, g, v, lr, momentum, w_bf16=None, stream=None):
    _check(load().sgd_momentum_step(_ptr(w), _ptr(g), _ptr(v), _ptr(w_bf16), w.numel(), lr,
                                    momentum, _stream(stream)), "sgd_momentum_step")


def mlp_gemm(A, B, C, M, N, K, a_trans=False, b_trans=False, bias=None, act=MLP_ACT_NONE,
             mask=None, stream=None):
    """C = epilogue(op(A) @ op(B)); tensors are 2-D row-major with unit inner stride."""
    in_dtype = _dtype_code(A)
    _check(load().mlp_gemm(M, N, K, _ptr(A), A.stride(0), int(a_trans), _ptr(B), B.stride(0),
                           int(b_trans), in_dtype, _ptr(bias), act, _ptr(mask),
                           mask.stride(0) if mask is not None else 0, _ptr(C), C.stride(0),
                           _dtype_code(C), _stream(stream)), "mlp_gemm")


def mlp_colsum_workspace_bytes(rows: int, cols: int) -> int:
    return load().mlp_colsum_workspace_bytes(rows, cols)


def mlp_colsum(X, out, rows=None, cols=None, workspace=None, stream=None):
    r = X.shape[0] if rows is None else rows
    c = out.shape[0] if cols is None else cols
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().mlp_colsum(_ptr(X), _dtype_code(X), r, c, X.stride(0), _ptr(out),
                             _ptr(workspace), wsb, _stream(stream)), "mlp_colsum")


def mse_workspace_bytes(n: int) -> int:
    return load().mse_workspace_bytes(n)


def mse_loss_fwd_bwd(y, t, loss_out, dy, workspace, stream=None):
    wsb = workspace.numel() * workspace.element_size()
    _check(load().mse_loss_fwd_bwd(_ptr(y), _ptr(t), y.numel(), _ptr(loss_out), _ptr(dy),
                                   _ptr(workspace), wsb, _stream(stream)), "mse_loss_fwd_bwd")


# ------------------------------------------------------------------ block

def mlp_block_workspace_bytes(T: int, d: int, hidden: int) -> int:
    return load().mlp_block_workspace_bytes(T, d, hidden)


def mlp_block_fwd(x, w_gate, w_down, y, rstd, eps=1e-6, slope=0.5, stream=None):
    T, d = x.shape
    h = w_gate.shape[1]
    _check(load().mlp_block_fwd(_ptr(x), _ptr(w_gate), _ptr(w_down), T, d, h, eps, slope,
                                _ptr(y), _ptr(rstd), _stream(stream)), "mlp_block_fwd")


def mlp_block_bwd(x, rstd, w_gate, w_down, dy, dx, dw_gate, dw_down, workspace, eps=1e-6,
                  slope=0.5, stream=None):
    T, d = x.shape
    h = w_gate.shape[1]
    wsb = workspace.numel() * workspace.element_size()
    _check(load().mlp_block_bwd(_ptr(x), _ptr(rstd), _ptr(w_gate), _ptr(w_down), _ptr(dy), T, d,
                                h, eps, slope, _ptr(dx), _ptr(dw_gate), _ptr(dw_down),
                                _ptr(workspace), wsb, _stream(stream)), "mlp_block_bwd")


def mlp_attn_prep_fwd(x, w_qkv, q_gain, qkv_out, rstd_out, n_q_heads, n_kv_heads,
                      rope_dims, seq_len, eps=1e-6, rope_theta=10000.0, head_dim=64, stream=None):
    """Fused RMSNorm -> QKV projection -> QK norm -> partial RoPE -> q gain."""
    T, d = x.shape
    _check(load().mlp_attn_prep_fwd(_ptr(x), _ptr(w_qkv), _ptr(q_gain), T, d, n_q_heads,
                                    n_kv_heads, head_dim, rope_dims, seq_len, eps, rope_theta,
                                    _ptr(qkv_out), _ptr(rstd_out), _stream(stream)),
           "mlp_attn_prep_fwd")


def mlp_stack_param_count(n_blocks: int, d: int, hidden: int) -> int:
    return load().mlp_stack_param_count(n_blocks, d, hidden)


def mlp_stack_workspace_bytes(n_blocks: int, T: int, d: int, hidden: int) -> int:
    return load().mlp_stack_workspace_bytes(n_blocks, T, d, hidden)


def mlp_stack_train_step(n_blocks, T, d, hidden, x0, target, params, velocity, grads,
                         params_bf16, lr, momentum, loss_out, workspace, eps=1e-6, slope=0.5,
                         stream=None):
    wsb = workspace.numel() * workspace.element_size()
    _check(load().mlp_stack_train_step(n_blocks, T, d, hidden, eps, slope, _ptr(x0), _ptr(target),
                                       _ptr(params), _ptr(velocity), _ptr(grads),
                                       _ptr(params_bf16), lr, momentum, _ptr(loss_out),
                                       _ptr(workspace), wsb, _stream(stream)),
           "mlp_stack_train_step")
