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


def rel_round(dtype) -> float:
    """Unit roundoff of round-to-nearest in the 16-bit type P and O are
    stored in: 2^-p for p significant bits (bf16: 8, fp16: 11)."""
    return 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -11


def o_tolerance(o_ref: np.ndarray, a_ref: np.ndarray, dtype) -> np.ndarray:
    """Per-element bound on |O_gpu - O|.

    The kernel rounds each probability p_k to the 16-bit type before the P V
    product (relative error <= r) while the row sum l uses the fp32 p_k, so
    O_gpu = sum_k w_k (1 + e_k) v_k with |e_k| <= r, i.e. an error of at most
    r * sum_k w_k |v_k| = r * a_ref (a_ref: the oracle's attention output on
    |V|), plus the final rounding of O (<= r |O|).  The tolerance is the
    method's 2e-3 bar, or this bound (+1e-5 for fp32 accumulation and the
    exp2 approximation) where the formats alone can exceed 2e-3 -- rows that
    average only a few keys."""
    r = rel_round(dtype)
    return np.maximum(TOL_O, r * (np.abs(a_ref) + np.abs(o_ref)) + 1e-5)


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


def assert_close_o(o_gpu: np.ndarray, o_ref: np.ndarray, a_ref: np.ndarray, dtype, what=""):
    tol = o_tolerance(o_ref, a_ref, dtype)
    err = np.abs(o_gpu.astype(np.float64) - o_ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} elements over tolerance; max err "
                           f"{err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")


def assert_close_lse(lse_gpu, lse_ref, what=""):
    err = max_err(lse_gpu, lse_ref)
    assert err <= TOL_LSE, f"{what}: max |dLSE| {err:.3e}"


def oracle_dense(q, k, v, scale, causal):
    """(O, lse, A) where A is the oracle output on |V| (for the tolerance)."""
    o, lse = oracle.attention(q, k, v, scale, causal, nthreads=threads())
    a, _ = oracle.attention(q, k, v.abs(), scale, causal, nthreads=threads())
    return o, lse, a


def oracle_varlen(q, k, v, cu, scale, causal):
    o, lse = oracle.attention_varlen(q, k, v, cu, scale, causal, nthreads=threads())
    a, _ = oracle.attention_varlen(q, k, v.abs(), cu, scale, causal, nthreads=threads())
    return o, lse, a
