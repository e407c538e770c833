"""Dense, non-causal shapes whose tile count leaves the last wave of the
persistent grid at most half full.  The last tiles then run as two key
halves, each writing O / l in fp32 and its lse, and a merge kernel combines
them (lse = log(e^lse0 + e^lse1), O = sum_i e^(lse_i - lse) O_i: the
running-softmax merge over disjoint key sets of the "Fused attention
kernel" card, Implementation sketch).  Parity against the fp64 oracle on
rows of split tiles and of whole tiles: 16-bit at d = 64 and 128, with an
additive bias, and e4m3 on its own dequantised inputs."""
import math

import numpy as np
import pytest
import torch

import attention_forward_softmax_gb300 as agb
import oracle
from datagen import normal, random_signs
from tests._gpu_helpers import TOL_LSE, n_eff, o_tolerance, qkv, threads
from tests.test_gpu_bias import run as run_bias
from tests.test_gpu_fp8 import fp8_forward, outlier_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    agb.build()
    agb.lib()


def split_shape(N):
    """(H, first split tile, tiles) for B = 1: the smallest head count whose
    tile count leaves 0 < rem <= grid / 2 tiles for the last wave."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nqt = (N + 255) // 256
    for H in range(sms // nqt + 1, 4 * sms):
        T = H * nqt
        grid = min(T, sms)
        rem = T % grid
        if 0 < 2 * rem <= grid:
            return H, T - rem, T
    raise AssertionError("no split shape found")


def sample(N, H, first_split, seed):
    """Rows of split tiles (heads at and after the first split tile) and of
    whole tiles (head 0): tile edges, first and last rows, random rows."""
    nqt = (N + 255) // 256
    rng = np.random.default_rng(seed)
    toks, heads = [], []
    for h in sorted({0, first_split // nqt, H - 1}):
        edges = [0, 1, 127, 128, 255, 256, N // 2, N // 2 + 1, N // 2 + 127, N // 2 + 128,
                 N - 256, N - 129, N - 128, N - 1]
        for n in edges + [int(r) for r in rng.integers(0, N, 6)]:
            toks.append(n)
            heads.append(h)
    return np.array(toks, np.int64), np.array(heads, np.int32)


@pytest.mark.parametrize("dtype,d,grp", [(torch.bfloat16, 128, 1), (torch.float16, 128, 1),
                                         (torch.bfloat16, 64, 1), (torch.bfloat16, 128, 2)])
def test_split_tail_16bit(dtype, d, grp):
    N = 4096
    H, first_split, T = split_shape(N)
    q, _, _ = qkv(9100 + d, (1, N, H, d), dtype)
    _, k, v = qkv(9150 + d + grp, (1, N, H // grp, d), dtype)
    o, lse = agb.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=False)
    torch.cuda.synchronize()
    assert agb.get_status() == 0
    toks, heads = sample(N, H, first_split, 9101)
    cu = np.array([0, N], np.int32)
    q2, k2, v2 = (x[0].to(torch.float64).numpy() for x in (q, k, v))
    scale = 1 / math.sqrt(d)
    rows = lambda vv, sc: oracle.attention_rows_gqa(q2, k2, vv, cu, cu, sc, False, toks, heads,
                                                     threads())
    o_ref, lse_ref = rows(v2, scale)
    a_ref, _ = rows(np.abs(v2), scale)
    _, lse2 = rows(v2, 2 * scale)
    og = o.float().cpu().numpy()[0][toks, heads]
    lg = lse.cpu().numpy()[0][heads, toks]
    tol = o_tolerance(o_ref, a_ref, dtype, n_eff(lse_ref, lse2)[:, None])
    err = np.abs(og - o_ref)
    print(f"split tail d={d} {dtype} H/H_kv={grp}: H={H}, {T} tiles, split from {first_split}: "
          f"max |dO| {err.max():.3e}, max |dlse| {np.abs(lg - lse_ref).max():.3e}")
    assert np.all(err <= tol), float((err - tol).max())
    assert float(np.abs(lg - lse_ref).max()) <= TOL_LSE


def test_split_tail_with_bias():
    """A per-head key bias, broadcast over rows, on a short shape with a
    split last wave (the whole output against the oracle)."""
    N, d = 512, 64
    H, first_split, T = split_shape(N)
    q, k, v = qkv(9200, (1, N, H, d), torch.bfloat16)
    bias = normal(9200, 5, (1, H, 1, N)).astype(np.float32)
    run_bias(q, k, v, bias, False, torch.bfloat16)


def test_split_tail_e4m3():
    """The e4m3 kernel with a split last wave, against the oracle run on the
    dequantised inputs it sees, row by row, within the bound of the e4m3
    arithmetic test (each half quantises P against its own maximum, so the
    same per-element bound holds for the merged rows); lse gets 2^-20 more
    for the fp32 merge."""
    N, d = 4096, 128
    H, first_split, T = split_shape(N)
    q, k, v = outlier_qkv(9300, (1, N, H, d))
    o, lse, (q8, k8, v8, dq, dk, dv) = fp8_forward(q, k, v, random_signs(9300, d), False)
    dvn = dv.cpu().numpy()
    qd = oracle.dequantize(q8.cpu().numpy(), dq.cpu().numpy())[0]
    kd = oracle.dequantize(k8.cpu().numpy(), dk.cpu().numpy())[0]
    vd = oracle.dequantize(v8.cpu().numpy(), dvn)[0]
    toks, heads = sample(N, H, first_split, 9301)
    cu = np.array([0, N], np.int32)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle.attention_rows(qd, kd, vd, cu, scale, False, toks, heads, threads())
    a_ref, _ = oracle.attention_rows(qd, kd, np.abs(vd), cu, scale, False, toks, heads, threads())
    smax = np.array([(np.abs(qd[t, h]) @ np.abs(kd[:, h]).T).max() for t, h in zip(toks, heads)])
    lse_tol = (d * 2.0 ** -23 * scale * smax + 2.0 ** -21 + (N / 16 + 8) * 2.0 ** -24
               + 2.0 ** -20 + 1e-7)
    lg = lse[0][heads, toks]
    assert np.all(np.abs(lg - lse_ref) <= lse_tol), float((np.abs(lg - lse_ref) - lse_tol).max())
    # P is stored as e4m3(p w), w in [1, 8]: subnormal codes below 2^-6 are
    # off by at most 2^-10 / w
    w_min = np.maximum(1.0, 8.0 * dvn.min(axis=2) / dvn.max(axis=2))[0]     # [H]
    sub = (2.0 ** -10 / w_min[heads])[:, None] * np.abs(vd).sum(axis=0)[heads]
    tol = (2.0 ** -4 + 2.0 ** -8) * a_ref + 2.0 ** -7 * np.abs(o_ref) + sub + 1e-5
    err = np.abs(o[0][toks, heads] - o_ref)
    print(f"split tail e4m3: H={H}, {T} tiles, split from {first_split}: max |dO| "
          f"{err.max():.3e}, max |dlse| {np.abs(lg - lse_ref).max():.3e}")
    assert np.all(err <= tol), float((err - tol).max())
