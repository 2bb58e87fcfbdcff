"""Python access to the fp64 CPU oracle (oracle/oracle.cpp).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the bench's
CPU-baseline leg are the only callers.  The product path never imports this
package.  The oracle shares no code with the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_F = ctypes.POINTER(ctypes.c_float)
_I = ctypes.POINTER(ctypes.c_int)
_L = ctypes.POINTER(ctypes.c_longlong)


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (fp64, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["g++", "-std=c++17", "-O3", "-fopenmp", "-ffp-contract=off",
                               "-fno-fast-math", "-shared", "-fPIC", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_LIB)
        L = _lib
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_max_threads.restype = ctypes.c_int
        L.orc_round_bf16.restype = ctypes.c_double
        L.orc_round_bf16.argtypes = [ctypes.c_double]
        L.orc_round_f16.restype = ctypes.c_double
        L.orc_round_f16.argtypes = [ctypes.c_double]
        L.orc_matmul_f32_linear.argtypes = [_F, ctypes.c_int, _F, ctypes.c_int,
                                            ctypes.c_longlong, ctypes.c_longlong,
                                            ctypes.c_longlong, _F, ctypes.c_int, _F,
                                            ctypes.c_longlong, _F]
        L.orc_colsum_f32_linear.argtypes = [_F, ctypes.c_longlong, ctypes.c_longlong,
                                            ctypes.c_longlong, _F]
        L.orc_attn_prep.argtypes = [_D, _D, _D, ctypes.c_longlong, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_longlong,
                                    ctypes.c_double, ctypes.c_double, _D]
        L.orc_attn_prep_rows_f32.argtypes = [_F, _F, _F, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_longlong, ctypes.c_double, ctypes.c_double,
                                             _L, ctypes.c_longlong, _D]
        L.orc_param_count.restype = ctypes.c_longlong
        L.orc_param_count.argtypes = [_I, ctypes.c_int]
        L.orc_matmul.argtypes = [_D, ctypes.c_int, _D, ctypes.c_int, ctypes.c_longlong,
                                 ctypes.c_longlong, ctypes.c_longlong, _D]
        L.orc_matmul_entries_f32.argtypes = [_F, ctypes.c_int, _F, ctypes.c_int,
                                             ctypes.c_longlong, ctypes.c_longlong,
                                             ctypes.c_longlong, _L, _L, ctypes.c_longlong, _D]
        L.orc_mlp_forward.argtypes = [_I, ctypes.c_int, _D, _D, ctypes.c_longlong, ctypes.c_int,
                                      _D, _D]
        L.orc_softmax_xent.argtypes = [_D, _I, ctypes.c_longlong, ctypes.c_int, ctypes.c_longlong,
                                       _D, _D, _D, _I]
        L.orc_mlp_backward.argtypes = [_I, ctypes.c_int, _D, _D, ctypes.c_longlong, _D, _D,
                                       ctypes.c_int, _D, _D]
        L.orc_colsum_f32.argtypes = [_F, ctypes.c_longlong, ctypes.c_longlong, ctypes.c_longlong,
                                     _D]
        L.orc_sgd_momentum.argtypes = [_D, _D, _D, ctypes.c_longlong, ctypes.c_double,
                                       ctypes.c_double]
        L.orc_mlp_train_step.restype = ctypes.c_double
        L.orc_mlp_train_step.argtypes = [_I, ctypes.c_int, _D, _D, _D, _I, ctypes.c_longlong,
                                         ctypes.c_double, ctypes.c_double, ctypes.c_int, _D]
        L.orc_mlp_forward_rows_f32.argtypes = [_I, ctypes.c_int, _F, _F, _L, ctypes.c_longlong,
                                               ctypes.c_int, _D]
        L.orc_block_fwd.argtypes = [_D, _D, _D, ctypes.c_longlong, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_double, ctypes.c_double, _D, _D]
        L.orc_block_bwd.argtypes = [_D, _D, _D, _D, ctypes.c_longlong, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_double, ctypes.c_double, _D, _D, _D]
        L.orc_block_fwd_rows_f32.argtypes = [_F, _F, _F, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_double, ctypes.c_double, _L,
                                             ctypes.c_longlong, _D, _D]
        L.orc_block_bwd_dx_rows_f32.argtypes = [_F, _F, _F, _F, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_double, ctypes.c_double, _L,
                                                ctypes.c_longlong, _D]
        L.orc_block_bwd_dw_entries_f32.argtypes = [_F, _F, _F, _F, ctypes.c_longlong,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                   ctypes.c_double, _I, _L, _L,
                                                   ctypes.c_longlong, _D]
        L.orc_mse.argtypes = [_D, _D, ctypes.c_longlong, _D, _D]
        L.orc_stack_fwd_bwd.restype = ctypes.c_double
        L.orc_stack_fwd_bwd.argtypes = [_D, _D, ctypes.c_int, ctypes.c_longlong, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_double, ctypes.c_double, _D, _D, _D]
    return _lib


# ----------------------------------------------------------------- wrappers

def _d(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _f(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _p(a, t):
    return None if a is None else a.ctypes.data_as(t)


def _dims(dims):
    return (ctypes.c_int * len(dims))(*dims), len(dims)


def set_threads(n: int) -> None:
    """Threads of the oracle's OpenMP loops (for timing)."""
    lib().orc_set_threads(int(n))


def max_threads() -> int:
    return lib().orc_max_threads()


def round_bf16(v: float) -> float:
    return lib().orc_round_bf16(float(v))


def round_f16(v: float) -> float:
    """Nearest IEEE binary16 value of v (ties to even, subnormals, overflow to
    infinity), as a float."""
    return lib().orc_round_f16(float(v))


def _points(bf16_points=False, points=None):
    """Rounding-points code of the oracle's MLP functions: 0 exact, 1 bf16
    points, 2 fp16 points (points: None, 0/1/2, "bf16" or "f16")."""
    if points is None:
        return 1 if bf16_points else 0
    if isinstance(points, str):
        return {"exact": 0, "bf16": 1, "f16": 2, "fp16": 2}[points]
    return int(points)


def param_count(dims) -> int:
    d, n = _dims(dims)
    return lib().orc_param_count(d, n)


def matmul(A, B, a_t=False, b_t=False):
    A, B = _d(A), _d(B)
    M = A.shape[1] if a_t else A.shape[0]
    K = A.shape[0] if a_t else A.shape[1]
    N = B.shape[0] if b_t else B.shape[1]
    C = np.empty((M, N))
    lib().orc_matmul(_p(A, _D), int(a_t), _p(B, _D), int(b_t), M, N, K, _p(C, _D))
    return C


def matmul_entries(A, B, ii, jj, a_t=False, b_t=False):
    A, B = _f(A), _f(B)
    M = A.shape[1] if a_t else A.shape[0]
    K = A.shape[0] if a_t else A.shape[1]
    N = B.shape[0] if b_t else B.shape[1]
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    out = np.empty(len(ii))
    lib().orc_matmul_entries_f32(_p(A, _F), int(a_t), _p(B, _F), int(b_t), M, N, K,
                                 _p(ii, _L), _p(jj, _L), len(ii), _p(out, _D))
    return out


def mlp_forward(dims, params, X, bf16_points=False, points=None):
    """Returns (list of hidden activations, logits Z)."""
    params, X = _d(params), _d(X)
    B = X.shape[0]
    n_act = sum(B * dims[l] for l in range(1, len(dims) - 1))
    acts = np.empty(max(n_act, 1))
    Z = np.empty((B, dims[-1]))
    d, n = _dims(dims)
    lib().orc_mlp_forward(d, n, _p(params, _D), _p(X, _D), B, _points(bf16_points, points),
                          _p(acts, _D), _p(Z, _D))
    hs, off = [], 0
    for l in range(1, len(dims) - 1):
        hs.append(acts[off:off + B * dims[l]].reshape(B, dims[l]))
        off += B * dims[l]
    return hs, Z


def softmax_xent(Z, y, B_norm=None):
    """Returns (mean loss, per-row loss, dZ, argmax)."""
    Z = _d(Z)
    B, C = Z.shape
    y = np.ascontiguousarray(y, dtype=np.int32)
    loss = np.zeros(1)
    rl = np.empty(B)
    dZ = np.empty((B, C))
    am = np.empty(B, dtype=np.int32)
    lib().orc_softmax_xent(_p(Z, _D), _p(y, _I), B, C, B if B_norm is None else B_norm,
                           _p(loss, _D), _p(rl, _D), _p(dZ, _D), _p(am, _I))
    return loss[0], rl, dZ, am


def mlp_backward(dims, params, X, hs, dZ, bf16_points=False, want_dx=False, points=None):
    params, X, dZ = _d(params), _d(X), _d(dZ)
    B = X.shape[0]
    acts = _d(np.concatenate([h.ravel() for h in hs])) if hs else np.zeros(1)
    g = np.empty(param_count(dims))
    dX = np.empty_like(X) if want_dx else None
    d, n = _dims(dims)
    lib().orc_mlp_backward(d, n, _p(params, _D), _p(X, _D), B, _p(acts, _D), _p(dZ, _D),
                           _points(bf16_points, points), _p(g, _D), _p(dX, _D))
    return (g, dX) if want_dx else g


def matmul_f32_linear(A, B, a_t=False, b_t=False, bias=None, act=0, mask=None):
    """fp32 C = act(chain + bias) with each chain one fused-multiply-add
    sequence over ascending k (the linear-order mode); mask keeps C > 0 cells.
    A is [M][K] (a_t False) or [K][M]; B is [K][N] (b_t False) or [N][K]."""
    A, B = _f(A), _f(B)
    Mr, K = (A.shape[1], A.shape[0]) if a_t else A.shape
    N = B.shape[0] if b_t else B.shape[1]
    C = np.empty((Mr, N), dtype=np.float32)
    bias = None if bias is None else _f(bias)
    mask = None if mask is None else _f(mask)
    lib().orc_matmul_f32_linear(_p(A, _F), int(a_t), _p(B, _F), int(b_t), Mr, N, K,
                                _p(bias, _F), int(act), _p(mask, _F),
                                0 if mask is None else mask.shape[1], _p(C, _F))
    return C


def colsum_f32_linear(X):
    """fp32 column sums, rows added in ascending order from 0."""
    X = _f(X)
    out = np.empty(X.shape[1], dtype=np.float32)
    lib().orc_colsum_f32_linear(_p(X, _F), X.shape[0], X.shape[1], X.shape[1], _p(out, _F))
    return out


def colsum(X):
    X = _f(X)
    out = np.empty(X.shape[1])
    lib().orc_colsum_f32(_p(X, _F), X.shape[0], X.shape[1], X.shape[1], _p(out, _D))
    return out


def sgd_momentum(w, g, v, lr, momentum):
    """Returns updated (w, v) as new arrays."""
    w, g, v = _d(w).copy(), _d(g), _d(v).copy()
    lib().orc_sgd_momentum(_p(w, _D), _p(g, _D), _p(v, _D), w.size, lr, momentum)
    return w, v


def mlp_train_step(dims, params, velocity, X, y, lr, momentum, bf16_points=False, points=None):
    """One step; returns (loss, new params, new velocity, grads)."""
    p, v = _d(params).copy(), _d(velocity).copy()
    X = _d(X)
    y = np.ascontiguousarray(y, dtype=np.int32)
    g = np.empty(p.size)
    d, n = _dims(dims)
    loss = lib().orc_mlp_train_step(d, n, _p(p, _D), _p(v, _D), _p(X, _D), _p(y, _I),
                                    X.shape[0], lr, momentum, _points(bf16_points, points),
                                    _p(g, _D))
    return loss, p, v, g


def mlp_forward_rows(dims, params, X, rows, bf16_points=False, points=None):
    params, X = _f(params), _f(X)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    Z = np.empty((len(rows), dims[-1]))
    d, n = _dims(dims)
    lib().orc_mlp_forward_rows_f32(d, n, _p(params, _F), _p(X, _F), _p(rows, _L), len(rows),
                                   _points(bf16_points, points), _p(Z, _D))
    return Z


def block_fwd(x, Wg, Wd, eps, slope):
    x, Wg, Wd = _d(x), _d(Wg), _d(Wd)
    T, d = x.shape
    h = Wg.shape[1]
    y = np.empty_like(x)
    r = np.empty(T)
    lib().orc_block_fwd(_p(x, _D), _p(Wg, _D), _p(Wd, _D), T, d, h, eps, slope,
                        _p(y, _D), _p(r, _D))
    return y, r


def block_bwd(x, Wg, Wd, dy, eps, slope):
    x, Wg, Wd, dy = _d(x), _d(Wg), _d(Wd), _d(dy)
    T, d = x.shape
    h = Wg.shape[1]
    dx = np.empty_like(x)
    dWg = np.empty((d, h))
    dWd = np.empty((h, d))
    lib().orc_block_bwd(_p(x, _D), _p(Wg, _D), _p(Wd, _D), _p(dy, _D), T, d, h, eps, slope,
                        _p(dx, _D), _p(dWg, _D), _p(dWd, _D))
    return dx, dWg, dWd


def block_fwd_rows(x, Wg, Wd, rows, eps, slope):
    x, Wg, Wd = _f(x), _f(Wg), _f(Wd)
    d = x.shape[1]
    h = Wg.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    y = np.empty((len(rows), d))
    r = np.empty(len(rows))
    lib().orc_block_fwd_rows_f32(_p(x, _F), _p(Wg, _F), _p(Wd, _F), d, h, eps, slope,
                                 _p(rows, _L), len(rows), _p(y, _D), _p(r, _D))
    return y, r


def block_bwd_dx_rows(x, Wg, Wd, dy, rows, eps, slope):
    x, Wg, Wd, dy = _f(x), _f(Wg), _f(Wd), _f(dy)
    d = x.shape[1]
    h = Wg.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    dx = np.empty((len(rows), d))
    lib().orc_block_bwd_dx_rows_f32(_p(x, _F), _p(Wg, _F), _p(Wd, _F), _p(dy, _F), d, h, eps,
                                    slope, _p(rows, _L), len(rows), _p(dx, _D))
    return dx


def block_bwd_dw_entries(x, Wg, Wd, dy, which, ii, jj, eps, slope):
    x, Wg, Wd, dy = _f(x), _f(Wg), _f(Wd), _f(dy)
    T, d = x.shape
    h = Wg.shape[1]
    which = np.ascontiguousarray(which, dtype=np.int32)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    out = np.empty(len(ii))
    lib().orc_block_bwd_dw_entries_f32(_p(x, _F), _p(Wg, _F), _p(Wd, _F), _p(dy, _F), T, d, h,
                                       eps, slope, _p(which, _I), _p(ii, _L), _p(jj, _L),
                                       len(ii), _p(out, _D))
    return out


def mse(y, t):
    y, t = _d(y), _d(t)
    loss = np.zeros(1)
    dy = np.empty_like(y)
    lib().orc_mse(_p(y, _D), _p(t, _D), y.size, _p(loss, _D), _p(dy, _D))
    return loss[0], dy


def stack_fwd_bwd(x0, params, n_blocks, d, h, eps, slope, target):
    x0, params, target = _d(x0), _d(params), _d(target)
    T = x0.shape[0]
    g = np.empty_like(params)
    dx0 = np.empty_like(x0)
    loss = lib().orc_stack_fwd_bwd(_p(x0, _D), _p(params, _D), n_blocks, T, d, h, eps, slope,
                                   _p(target, _D), _p(g, _D), _p(dx0, _D))
    return loss, g, dx0


def attn_prep(x, W, q_gain, n_q, n_kv, hd, rope_dims, seq_len, eps=1e-6, theta=10000.0):
    """Fused attention preprocessing of every token: RMSNorm, QKV projection,
    QK norm, partial RoPE, q gain; returns [T][(n_q + 2 n_kv) hd]."""
    x, W, g = _d(x), _d(W), _d(q_gain)
    T, d = x.shape
    out = np.empty((T, (n_q + 2 * n_kv) * hd))
    lib().orc_attn_prep(_p(x, _D), _p(W, _D), _p(g, _D), T, d, n_q, n_kv, hd, rope_dims,
                        seq_len, eps, theta, _p(out, _D))
    return out


def attn_prep_rows(x, W, q_gain, rows, n_q, n_kv, hd, rope_dims, seq_len, eps=1e-6,
                   theta=10000.0):
    """attn_prep for the listed rows only (fp32 inputs as stored)."""
    x, W, g = _f(x), _f(W), _f(q_gain)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((len(rows), (n_q + 2 * n_kv) * hd))
    lib().orc_attn_prep_rows_f32(_p(x, _F), _p(W, _F), _p(g, _F), x.shape[1], n_q, n_kv, hd,
                                 rope_dims, seq_len, eps, theta, _p(rows, _L), len(rows),
                                 _p(out, _D))
    return out

