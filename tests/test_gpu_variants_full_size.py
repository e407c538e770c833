"""GPU parity of the inference variants at the sizes bench.py times them, in
the same launch configuration: the causal grouped-K/V-head workload (B=4,
H=32, H_kv=8, N=8192, d=128) on sampled rows, and paged decoding (32
sequences of 512-8192 cached positions, one new query each, H=32, H_kv=8,
64-token pages in a shuffled order, automatic split count) on every output
row.  Element by element against the fp64 oracle, with the tolerance rule
of the other 16-bit tests (the bare 2e-3 where at least 64 keys carry the
row's weight and |O| < 0.5)."""
import math

import numpy as np
import pytest
import torch

import attention_forward_softmax_gb300 as agb
import oracle
from datagen import workloads as W
from tests._gpu_helpers import (TOL_LSE, TOL_O, assert_close_o, n_eff, o_tolerance,
                                sample_rows, threads)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    agb.build()
    agb.lib()


def test_gqa_causal_bench_workload_sampled_rows():
    w = W.gqa_causal()
    x = W.make_inputs(w)
    q, k, v = (x[n].cuda() for n in "qkv")
    o, lse = agb.attn_fwd(q, k, v, causal=w.causal)
    torch.cuda.synchronize()
    assert agb.get_status() == 0
    rng = np.random.default_rng(w.seed + 50)
    ns = sample_rows(w.N, 96, w.seed + 51)
    bs = rng.integers(0, w.B, size=len(ns))
    toks = (bs * w.N + ns).astype(np.int64)
    heads = rng.integers(0, w.H, size=len(toks)).astype(np.int32)
    cu = w.cu_seqlens()
    qf = x["q"].to(torch.float64).numpy().reshape(w.tokens, w.H, w.d)
    kf = x["k"].to(torch.float64).numpy().reshape(w.tokens, w.Hkv, w.d)
    vf = x["v"].to(torch.float64).numpy().reshape(w.tokens, w.Hkv, w.d)
    args = (cu, cu)
    o_ref, lse_ref = oracle.attention_rows_gqa(qf, kf, vf, *args, w.scale, True, toks, heads,
                                               threads())
    a_ref, _ = oracle.attention_rows_gqa(qf, kf, np.abs(vf), *args, w.scale, True, toks, heads,
                                         threads())
    _, lse2 = oracle.attention_rows_gqa(qf, kf, vf, *args, 2 * w.scale, True, toks, heads,
                                        threads())
    og = o.float().cpu().numpy().reshape(w.tokens, w.H, w.d)[toks, heads]
    lg = lse.cpu().numpy()[bs, heads, ns]
    tol = o_tolerance(o_ref, a_ref, torch.bfloat16, n_eff(lse_ref, lse2)[:, None])
    err = np.abs(og - o_ref)
    strict = tol == TOL_O
    print(f"{w.name}: {len(toks)} rows, max |dO| {err.max():.3e} (bare 2e-3 on "
          f"{strict.mean():.0%} of elements), max |dlse| {np.abs(lg - lse_ref).max():.3e}")
    assert np.all(err <= tol), float((err - tol).max())
    assert float(np.abs(lg - lse_ref).max()) <= TOL_LSE


def test_paged_decode_bench_workload_all_rows():
    w = W.paged_decode()
    x = W.make_paged_inputs(w)
    q = x["q"]
    kc, vc = x["k_cache"], x["v_cache"]
    table, seql = x["block_table"], x["seqlens"]
    o, lse = agb.attn_fwd_paged(q.cuda(), kc.cuda(), vc.cuda(), torch.from_numpy(table).cuda(),
                                torch.from_numpy(seql).cuda(), max(w.lengths), causal=w.causal)
    torch.cuda.synchronize()
    assert agb.get_status() == 0
    lens = [int(v) for v in seql]
    scale = 1 / math.sqrt(w.d)
    o_ref, lse_ref = oracle.attention_paged(q, kc, vc, table, lens, scale, w.causal, threads())
    a_ref, _ = oracle.attention_paged(q, kc, vc.abs(), table, lens, scale, w.causal, threads())
    _, lse2 = oracle.attention_paged(q, kc, vc, table, lens, 2 * scale, w.causal, threads())
    og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
    ne = n_eff(lse_ref, lse2).transpose(0, 2, 1)[..., None]
    assert_close_o(og, o_ref, a_ref, torch.bfloat16, ne, "paged decode workload")
    assert float(np.abs(lg - lse_ref).max()) <= TOL_LSE
