"""Shared helpers of the GPU parity tests (tolerances, conversions)."""
import numpy as np
import torch


def bf16_values(a):
    """float64 copy of a float array after rounding to bf16 (what the GPU receives)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16) \
        .double().numpy()


def f16_values(a):
    """float64 copy of a float array after rounding to IEEE binary16."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.float16) \
        .double().numpy()


def values16(a, dtype):
    """float64 copy of a float array after rounding to the 16-bit torch dtype."""
    return f16_values(a) if dtype == torch.float16 else bf16_values(a)


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def rel_to_max(got, ref):
    """max |got - ref| / max |ref| (the per-tensor bf16-path error measure)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    return np.abs(got - ref).max() / (den if den > 0 else 1.0)


def assert_elementwise(got, ref, rtol, atol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        i = np.argmax(err - (atol + rtol * np.abs(ref)))
        raise AssertionError("%s: %d / %d elements out of tolerance; worst at %d: got %r ref %r"
                             % (what, bad.sum(), bad.size, i, got.ravel()[i], ref.ravel()[i]))


def near_tie_rows(Z, rel=1e-6):
    """Rows whose top-2 logits differ by less than rel * |max| (argmax not unique enough)."""
    s = np.sort(np.asarray(Z, dtype=np.float64), axis=1)
    gap = s[:, -1] - s[:, -2]
    return gap < rel * np.maximum(np.abs(s[:, -1]), 1e-30)
