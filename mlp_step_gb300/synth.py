"""Seeded synthetic inputs, shared by the CUDA path, the oracle tests and the bench.

This module holds no arithmetic of the training step: it only draws numbers.
Every draw comes from one counter-based generator, SplitMix64 (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014, with
Vigna's published finaliser constants), evaluated at an explicit counter, so a
value depends only on (seed, stream, index) and never on call order or on the
machine.

    key(seed, stream) = mix(seed * 0x9E3779B97F4A7C15 + stream)
    word(seed, stream, i) = mix(key + (i + 1) * 0x9E3779B97F4A7C15)

where mix is the SplitMix64 output function.  Derived draws:

* uniform01: top 24 bits of the word times 2**-24, in [0, 1)
* uniform integer in [0, n): (word >> 32) * n >> 32
* byte: word >> 56 (uniform 0..255)
* normal: Box-Muller cosine branch on the uniforms at counters 2i and 2i+1

The recipes (image bytes scaled by 1/255, labels uniform over the classes,
He-uniform weights U(-sqrt(6/fan_in), +sqrt(6/fan_in)), N(0, 0.02) block
weights, N(0, 1) activations) follow the workload descriptions of the 784-256-10
capstone ("Capstone 5: train a network with your CUDA kernels", "The minimum
model": seed 20260829, batch 128) and of the MLP block ("Full-Depth MLP
Megakernel", "What Worked"); the distributions themselves are the workload
definitions this library is measured on.
"""
from __future__ import annotations

import numpy as np

SEED = 20260829

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Stream ids: one per kind of draw so that no two tensors share counters.
STREAM_X = 1
STREAM_LABELS = 2
STREAM_W = 100          # + layer index
STREAM_BLOCK_X = 200
STREAM_BLOCK_WG = 300   # + block index
STREAM_BLOCK_WD = 400   # + block index
STREAM_BLOCK_DY = 500
STREAM_TARGET = 600
STREAM_GENERIC = 1000   # + caller-chosen offset, for kernel-level tests


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) * _GOLDEN + np.uint64(stream)
        return _mix(np.asarray(base, dtype=np.uint64))[()]


def words(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """n raw 64-bit words at counters start .. start+n-1."""
    key = _key(seed, stream)
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + idx * _GOLDEN)


def uniform01(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """float64 uniforms in [0, 1) with 24 bits of resolution."""
    w = words(seed, stream, n, start)
    return (w >> np.uint64(40)).astype(np.float64) * (1.0 / (1 << 24))


def randint(seed: int, stream: int, n: int, high: int) -> np.ndarray:
    w = words(seed, stream, n)
    return (((w >> np.uint64(32)) * np.uint64(high)) >> np.uint64(32)).astype(np.int32)


def bytes_u8(seed: int, stream: int, n: int) -> np.ndarray:
    return (words(seed, stream, n) >> np.uint64(56)).astype(np.uint8)


def normal(seed: int, stream: int, n: int, chunk: int = 1 << 22) -> np.ndarray:
    """float64 standard normals (Box-Muller, cosine branch)."""
    out = np.empty(n, dtype=np.float64)
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        u = uniform01(seed, stream, 2 * m, start=2 * s).reshape(m, 2)
        r = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
        out[s:s + m] = r * np.cos(2.0 * np.pi * u[:, 1])
    return out


# ---------------------------------------------------------------- recipes

def images_u8(batch: int, features: int = 784, seed: int = SEED, start_row: int = 0) -> np.ndarray:
    """uint8 images [batch, features], uniform 0..255 (28x28 byte format)."""
    w = words(seed, STREAM_X, batch * features, start=start_row * features)
    return (w >> np.uint64(56)).astype(np.uint8).reshape(batch, features)


def labels(batch: int, classes: int, seed: int = SEED, start_row: int = 0) -> np.ndarray:
    w = words(seed, STREAM_LABELS, batch, start=start_row)
    return (((w >> np.uint64(32)) * np.uint64(classes)) >> np.uint64(32)).astype(np.int32)


def he_uniform(fan_in: int, fan_out: int, layer: int, seed: int = SEED) -> np.ndarray:
    """float32 [fan_in, fan_out] drawn from U(-sqrt(6/fan_in), +sqrt(6/fan_in))."""
    a = np.sqrt(6.0 / fan_in)
    u = uniform01(seed, STREAM_W + layer, fan_in * fan_out)
    return ((2.0 * u - 1.0) * a).astype(np.float32).reshape(fan_in, fan_out)


def mlp_flat_params(dims, seed: int = SEED) -> np.ndarray:
    """Flat float32 parameters in the order W1, b1, W2, b2, ... (biases zero)."""
    parts = []
    for l in range(len(dims) - 1):
        parts.append(he_uniform(dims[l], dims[l + 1], l, seed).ravel())
        parts.append(np.zeros(dims[l + 1], dtype=np.float32))
    return np.concatenate(parts)


def uniform_f32(shape, stream: int, lo: float = -1.0, hi: float = 1.0,
                seed: int = SEED) -> np.ndarray:
    """float32 uniforms in [lo, hi) (cheaper than normals for very large tensors)."""
    n = int(np.prod(shape))
    u = uniform01(seed, stream, n)
    return (lo + (hi - lo) * u).astype(np.float32).reshape(shape)


def normal_f32(shape, stream: int, std: float = 1.0, seed: int = SEED) -> np.ndarray:
    n = int(np.prod(shape))
    return (normal(seed, stream, n) * std).astype(np.float32).reshape(shape)


def logits_pm60(batch: int, classes: int, seed: int = SEED):
    """Rows of logits drawn from {+60, -60}; each row has k >= 1 entries at +60.

    Returns (logits float32 [batch, classes], k per row int32).
    """
    k = 1 + randint(seed, STREAM_GENERIC + 7, batch, classes)
    u = uniform01(seed, STREAM_GENERIC + 8, batch * classes).reshape(batch, classes)
    order = np.argsort(u, axis=1, kind="stable")
    z = np.full((batch, classes), -60.0, dtype=np.float32)
    for b in range(batch):
        z[b, order[b, :k[b]]] = 60.0
    return z, k.astype(np.int32)
