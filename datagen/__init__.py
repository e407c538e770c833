"""Seeded synthetic inputs for the attention workloads.

This module draws random numbers and nothing else: it holds no attention,
softmax, rotation or quantisation arithmetic.  Both the CUDA path's tests and
the CPU oracle receive the same bytes from it.

Generator: a counter-based splitmix64 stream (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014; the 64-bit finaliser
published by Vigna).  Stream ``s`` under seed ``seed`` starts from the state
``mix(seed) ^ mix(s + 0x5851F42D4C957F2D)`` and advances by the golden-ratio
increment, so element ``i`` of a stream is ``mix(state0 + (i + 1) * G)``; any
element can be produced without the ones before it.  Uniforms take the top 53
bits, normals use the Box-Muller transform (both outputs of a pair).
"""
from __future__ import annotations

import numpy as np

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_SALT = 0x5851F42D4C957F2D
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser on a uint64 array (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _mix_scalar(x: int) -> int:
    return int(_mix(np.array([x & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0])


def _state0(seed: int, stream: int) -> int:
    return _mix_scalar(seed) ^ _mix_scalar(stream + _STREAM_SALT)


def bits(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """``n`` raw uint64 draws, elements ``offset .. offset+n-1`` of the stream."""
    s0 = np.uint64(_state0(seed, stream))
    out = np.empty(n, dtype=np.uint64)
    for a in range(0, n, _CHUNK):
        b = min(n, a + _CHUNK)
        idx = np.arange(offset + a + 1, offset + b + 1, dtype=np.uint64)
        with np.errstate(over="ignore"):
            out[a:b] = _mix(s0 + idx * _G)
    return out


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    """``n`` float64 uniforms in the open-closed interval (0, 1]."""
    u = bits(seed, stream, n)
    return ((u >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal(seed: int, stream: int, shape, dtype=np.float32) -> np.ndarray:
    """Standard normal draws of the given shape (Box-Muller on stream pairs)."""
    n = int(np.prod(shape))
    m = (n + 1) // 2
    out = np.empty(2 * m, dtype=np.float64)
    for a in range(0, m, _CHUNK):
        b = min(m, a + _CHUNK)
        u = bits(seed, stream, 2 * (b - a), offset=2 * a)
        u = ((u >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        r = np.sqrt(-2.0 * np.log(u[0::2]))
        t = (2.0 * np.pi) * u[1::2]
        out[2 * a:2 * b:2] = r * np.cos(t)
        out[2 * a + 1:2 * b:2] = r * np.sin(t)
    return out[:n].reshape(shape).astype(dtype)


def outlier_normal(seed: int, stream: int, shape, frac: float = 1e-3,
                   sigma: float = 10.0, dtype=np.float32) -> np.ndarray:
    """N(0,1) draws, each entry independently replaced with probability
    ``frac`` by a draw from N(0, sigma^2)."""
    x = normal(seed, stream, shape, dtype=np.float64)
    n = x.size
    pick = uniform(seed, stream + 1000, n).reshape(shape) <= frac
    big = sigma * normal(seed, stream + 2000, shape, dtype=np.float64)
    x[pick] = big[pick]
    return x.astype(dtype)


def random_signs(seed: int, d: int) -> np.ndarray:
    """``d`` independent fair signs as int8 (+1 / -1)."""
    b = bits(seed, 3000, d)
    return np.where((b >> np.uint64(63)) == 0, 1, -1).astype(np.int8)


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    """``n`` integers uniform on [lo, hi] inclusive."""
    u = bits(seed, stream, n) >> np.uint64(11)
    span = hi - lo + 1
    return (lo + np.floor(u.astype(np.float64) * (2.0 ** -53) * span)).astype(np.int64)


def to_bf16(x: np.ndarray):
    """Round float32 draws to bfloat16 (round-to-nearest-even), as a CPU torch
    tensor.  The bf16 bytes are what both the GPU and the oracle consume."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def to_fp16(x: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float16)
