"""Shared helpers for the GPU parity tests (inputs from datagen, expected
values from the oracle only)."""
import math
import os

import numpy as np
import torch

import oracle
from datagen import normal, to_bf16, to_fp16

# Tolerances stated by the method's parity bar for N(0,1) inputs.
TOL_O = 2e-3
TOL_LSE = 1e-3


def ulp_half(x: np.ndarray, mant_bits: int) -> np.ndarray:
    """Half a unit in the last place of |x| in a format with `mant_bits`
    explicit mantissa bits (bf16: 7, fp16: 10)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -14)))
    return 2.0 ** (e - mant_bits) / 2


def o_tolerance(o_ref: np.ndarray, dtype) -> np.ndarray:
    """2e-3, plus the output format's own half-ulp where |O| is large enough
    for rounding to exceed it (small N, where O is close to one V row)."""
    bits = 7 if dtype == torch.bfloat16 else 10
    return TOL_O + ulp_half(o_ref, bits)


def qkv(seed, shape, dtype):
    conv = to_bf16 if dtype == torch.bfloat16 else to_fp16
    return [conv(normal(seed, s, shape)) for s in range(3)]


def threads():
    return max(1, os.cpu_count() or 1)


def sample_rows(N: int, count: int, seed: int):
    """Rows 0, 1, N-1, N-2, the 128-row tile edges, plus seeded random rows."""
    base = {0, 1, N - 1, N - 2}
    for e in range(128, N, 128):
        base.update({e - 1, e})
    rng = np.random.default_rng(seed)
    extra = rng.integers(0, N, size=max(0, count - len(base)))
    rows = sorted(r for r in base.union(extra.tolist()) if 0 <= r < N)
    return np.array(rows, dtype=np.int64)


def max_err(a, b):
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64))))


def assert_close_o(o_gpu: np.ndarray, o_ref: np.ndarray, dtype, what=""):
    tol = o_tolerance(o_ref, dtype)
    err = np.abs(o_gpu.astype(np.float64) - o_ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} elements over tolerance; max err "
                           f"{err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")


def assert_close_lse(lse_gpu, lse_ref, what=""):
    err = max_err(lse_gpu, lse_ref)
    assert err <= TOL_LSE, f"{what}: max |dLSE| {err:.3e}"
