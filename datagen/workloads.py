"""Named synthetic attention workloads (shapes, seeds, value distributions).

Each workload is described by what it is and its sizes.  Inputs are drawn with
:mod:`datagen` and returned as CPU tensors; callers move them to the device.

Recipe (shared by tests, the benchmark and the oracle's timing sample):
  * Q, K, V entries are i.i.d. N(0, 1) float32 draws rounded to bf16 (or fp16),
    streams 0, 1, 2 of the workload's seed;
  * the fp8 workload replaces each entry independently with probability 1e-3 by
    an N(0, 10^2) draw (streams +1000 / +2000 of the same stream), and draws a
    random sign vector of length d for the Hadamard rotation;
  * the varlen workload draws 32 integer lengths uniform on [64, 4096]
    (stream 10) and packs the sequences back to back;
  * the backward workloads take the dense shape and add the upstream
    gradient dO, N(0, 1) draws of stream 9 rounded like Q.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

from . import normal, outlier_normal, random_signs, to_bf16, to_fp16, uniform_int


@dataclass
class Workload:
    name: str
    dtype: str            # "bf16", "fp16" or "fp8" (fp8: bf16 inputs quantised on device)
    B: int
    H: int
    N: int                # sequence length (dense); max length (varlen)
    d: int
    causal: bool
    seed: int
    lengths: Optional[List[int]] = None   # varlen only
    outliers: bool = False
    Hkv: Optional[int] = None             # K/V heads when fewer than H (grouped)

    @property
    def varlen(self) -> bool:
        return self.lengths is not None

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    @property
    def tokens(self) -> int:
        return int(sum(self.lengths)) if self.varlen else self.B * self.N

    def flops(self) -> float:
        """Attention-forward FLOP count 4*B*H*N^2*d, halved when causal; for
        varlen the per-sequence counts are summed."""
        if self.varlen:
            f = sum(4.0 * self.H * L * L * self.d for L in self.lengths)
        else:
            f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2.0 if self.causal else f

    def cu_seqlens(self) -> np.ndarray:
        if self.varlen:
            lens = np.asarray(self.lengths, dtype=np.int64)
        else:
            lens = np.full(self.B, self.N, dtype=np.int64)
        return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def _shape(w: Workload, heads=None):
    h = w.H if heads is None else heads
    return (w.tokens, h, w.d) if w.varlen else (w.B, w.N, h, w.d)


def make_inputs(w: Workload) -> dict:
    """Seeded Q, K, V (CPU tensors, bf16 or fp16; layout [B,N,H,d] dense or
    [T,H,d] packed), plus cu_seqlens (int32) and, for fp8, the sign vector."""
    conv = to_fp16 if w.dtype == "fp16" else to_bf16
    out = {}
    for s, nm in enumerate("qkv"):
        shape = _shape(w, None if nm == "q" else w.Hkv)
        if w.outliers:
            x = outlier_normal(w.seed, s, shape)
        else:
            x = normal(w.seed, s, shape)
        out[nm] = conv(x)
    out["cu_seqlens"] = w.cu_seqlens()
    if w.dtype == "fp8":
        out["signs"] = random_signs(w.seed, w.d)
    return out


def varlen_lengths(seed: int, nseq: int, lo: int, hi: int) -> List[int]:
    return [int(x) for x in uniform_int(seed, 10, nseq, lo, hi)]


# The five workloads the method is measured on.
TINY = Workload("bf16 non-causal B=1 H=1 N=128 d=64", "bf16", 1, 1, 128, 64, False, 1001)
DENSE = Workload("bf16 non-causal B=4 H=16 N=8448 d=128", "bf16", 4, 16, 8448, 128, False, 1002)
FP8 = Workload("fp8 e4m3 non-causal B=4 H=16 N=8192 d=128, 0.1% outliers",
               "fp8", 4, 16, 8192, 128, False, 1003, outliers=True)


def causal_sweep() -> List[Workload]:
    out = []
    for (H, d) in ((16, 128), (32, 64)):
        for N in (512, 1024, 2048, 4096, 8192, 16384):
            out.append(Workload(f"bf16 causal B={16384 // N} H={H} N={N} d={d}",
                                "bf16", 16384 // N, H, N, d, True, 1004))
    return out


def varlen_causal() -> Workload:
    lens = varlen_lengths(1005, 32, 64, 4096)
    return Workload("bf16 causal varlen 32 seqs L~U[64,4096] H=32 d=128", "bf16",
                    32, 32, max(lens), 128, True, 1005, lengths=lens)


def gqa_causal() -> Workload:
    """Grouped K/V heads (8 query heads per K/V head), causal prefill."""
    return Workload("bf16 causal GQA B=4 H=32 H_kv=8 N=8192 d=128", "bf16", 4, 32, 8192, 128,
                    True, 1006, Hkv=8)


@dataclass
class PagedWorkload:
    """Decoding against a paged K/V cache: each sequence has `lengths[b]`
    cached positions and Nq new queries."""
    name: str
    dtype: str
    lengths: List[int]
    Nq: int
    H: int
    Hkv: int
    d: int
    page_size: int
    causal: bool
    seed: int

    @property
    def B(self) -> int:
        return len(self.lengths)

    def flops(self) -> float:
        return sum(4.0 * self.H * self.Nq * L * self.d for L in self.lengths)

    def bytes(self) -> int:
        """Bytes a pass must move: every cached K and V row once, Q and O."""
        kv = sum(self.lengths) * self.Hkv * self.d * 2 * 2
        return kv + 2 * self.B * self.Nq * self.H * self.d * 2 + 4 * self.B * self.H * self.Nq


def paged_decode() -> PagedWorkload:
    lens = [int(x) for x in uniform_int(1007, 30, 32, 512, 8192)]
    return PagedWorkload("bf16 paged decode 32 seqs L~U[512,8192] Nq=1 H=32 H_kv=8 d=128 page=64",
                         "bf16", lens, 1, 32, 8, 128, 64, True, 1007)


def make_paged_inputs(w: PagedWorkload) -> dict:
    """q [B, Nq, H, d]; k_cache, v_cache [pages, page_size, H_kv, d] with the
    pages of all sequences handed out in a seeded random order (plus two
    spare pages); block_table int32 [B, max_pages]; seqlens int32 [B]."""
    conv = to_fp16 if w.dtype == "fp16" else to_bf16
    P = w.page_size
    need = [(L + P - 1) // P for L in w.lengths]
    npages = sum(need) + 2
    perm = np.argsort(uniform_int(w.seed, 31, npages, 0, 1 << 30), kind="stable")
    table = np.zeros((w.B, max(need)), dtype=np.int32)
    used = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[used:used + n]
        used += n
    return {"q": conv(normal(w.seed, 0, (w.B, w.Nq, w.H, w.d))),
            "k_cache": conv(normal(w.seed, 1, (npages, P, w.Hkv, w.d))),
            "v_cache": conv(normal(w.seed, 2, (npages, P, w.Hkv, w.d))),
            "block_table": table,
            "seqlens": np.asarray(w.lengths, dtype=np.int32)}


def backward(causal: bool) -> Workload:
    """The backward pass on the shape of the dense workload."""
    return Workload(f"bf16 backward {'causal' if causal else 'non-causal'} B=4 H=16 N=8448 d=128",
                    "bf16", 4, 16, 8448, 128, causal, 1008)


def make_dout(w: Workload):
    """Seeded upstream gradient dO, shaped and rounded like Q."""
    conv = to_fp16 if w.dtype == "fp16" else to_bf16
    return conv(normal(w.seed, 9, _shape(w)))
