"""GPU parity of the backward pass (attn_bwd) against the fp64 oracle's
gradients, element by element, on the kernel's own forward outputs: dense and
causal, grouped K/V heads, ragged tails, both 16-bit types.

Error bound per element (first order in the unit roundoff u of the 16-bit
type; P, dS and O are the only values the kernel rounds before using them):
  * dV = P^T dO with P rounded:            u (|P|^T |dO|)
  * dS = P (dP - D) rounded, and D = rowsum(dO * O) from the rounded O
    (|dD_i| <= u sum_c |dO_ic| |O_ic|):     |ddS| <= u |dS| + |P| |dD|
  * dK = scale dS^T Q, dQ = scale dS K:    scale (|ddS|^T |Q|), scale (|ddS| |K|)
plus the half-ulp of the rounded output and 1e-4 of the tensor's largest
value for fp32 accumulation order (dQ summed over key blocks by bulk
reductions in L2, in no fixed order) and the exp2 approximation.  |P|, |dS| for the bound are formed in float64 here; the
expected values come from the oracle."""
import math

import numpy as np
import pytest
import torch

import attention_forward_softmax_gb300 as agb
import oracle
from datagen import normal, to_bf16, to_fp16
from tests._gpu_helpers import half_ulp, qkv, rel_round, threads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    agb.build()
    agb.lib()


def bounds(q, k, v, do, scale, causal, u):
    """(|P|^T|dO|, |ddS|^T|Q|, |ddS||K|) per element, in [B, N, heads, d]."""
    q, k, v, do = (x.astype(np.float64) for x in (q, k, v, do))
    B, N, H, d = q.shape
    g = H // k.shape[2]
    kr, vr = np.repeat(k, g, axis=2), np.repeat(v, g, axis=2)
    s = np.einsum("bnhd,bmhd->bhnm", q, kr) * scale
    if causal:
        s = np.where(np.tril(np.ones((N, N), bool)), s, -np.inf)
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    o = np.einsum("bhnm,bmhd->bnhd", p, vr)
    dp = np.einsum("bnhd,bmhd->bhnm", do, vr)
    D = np.einsum("bnhd,bnhd->bhn", do, o)
    dD = u * np.einsum("bnhd,bnhd->bhn", np.abs(do), np.abs(o))
    ds = p * (dp - D[..., None])
    dds = u * np.abs(ds) + p * dD[..., None]
    bv = u * np.einsum("bhnm,bnhd->bmhd", p, np.abs(do))
    bk = scale * np.einsum("bhnm,bnhd->bmhd", dds, np.abs(q))
    bq = scale * np.einsum("bhnm,bmhd->bnhd", dds, np.abs(kr))
    def fold(x):   # sum the query heads of each K/V group
        return x.reshape(B, N, k.shape[2], g, d).sum(axis=3)
    return fold(bv), fold(bk), bq


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,H,Hkv,B", [(128, 2, 2, 2), (300, 4, 2, 2), (513, 3, 1, 2),
                                       (1100, 8, 2, 1)])
def test_backward_parity(N, H, Hkv, B, causal, dtype):
    d = 128
    conv = to_bf16 if dtype == torch.bfloat16 else to_fp16
    q, _, _ = qkv(8000 + N + H, (B, N, H, d), dtype)
    _, k, v = qkv(8100 + N + H, (B, N, Hkv, d), dtype)
    do = conv(normal(8200 + N, 7, (B, N, H, d)))
    scale = 1 / math.sqrt(d)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = agb.attn_fwd(qd, kd, vd, causal=causal)
    dq, dk, dv = agb.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal)
    torch.cuda.synchronize()
    assert agb.get_status() == 0
    rq, rk, rv = oracle.attention_backward(q, k, v, do, scale, causal, threads())
    u = rel_round(dtype)
    bv, bk, bq = bounds(*(x.float().numpy() for x in (q, k, v, do)), scale, causal, u)
    for name, got, ref, bnd in (("dv", dv, rv, bv), ("dk", dk, rk, bk), ("dq", dq, rq, bq)):
        g = got.float().cpu().numpy()
        tol = bnd + half_ulp(ref, dtype) + 1e-4 * np.abs(ref).max()
        err = np.abs(g - ref)
        print(f"{name}: max err {err.max():.3e}, max |ref| {np.abs(ref).max():.3e}")
        assert np.all(err <= tol), (name, float((err - tol).max()),
                                    np.unravel_index(np.argmax(err - tol), err.shape))


def test_backward_rejects_unsupported_head_size():
    q = torch.zeros((1, 16, 2, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 2, 16), dtype=torch.float32, device="cuda")
    with pytest.raises(agb.AttnError):
        agb.attn_bwd(q, q, q, q, lse, q)


def bounds_rows(q, k, v, do, scale, causal, u, qrows, krows, chunk=512):
    """The same first-order bound for selected rows of one sequence and head
    (q, k, v, do [L, d]), formed in float64 over query chunks so that a
    full-length sequence never needs an L x L array."""
    q, k, v, do = (x.astype(np.float64) for x in (q, k, v, do))
    L, d = q.shape
    kr = np.asarray(krows)
    bq = np.zeros((len(qrows), d))
    bk = np.zeros((len(kr), d))
    bv = np.zeros((len(kr), d))
    qpos = {int(i): n for n, i in enumerate(qrows)}
    for c0 in range(0, L, chunk):
        c1 = min(L, c0 + chunk)
        s = q[c0:c1] @ k.T * scale
        if causal:
            s = np.where(np.arange(L)[None, :] <= np.arange(c0, c1)[:, None], s, -np.inf)
        p = np.exp(s - s.max(-1, keepdims=True))
        p /= p.sum(-1, keepdims=True)
        o = p @ v
        D = (do[c0:c1] * o).sum(-1)
        dD = u * (np.abs(do[c0:c1]) * np.abs(o)).sum(-1)
        ds = p * (do[c0:c1] @ v.T - D[:, None])
        dds = u * np.abs(ds) + p * dD[:, None]
        bv += u * p[:, kr].T @ np.abs(do[c0:c1])
        bk += scale * dds[:, kr].T @ np.abs(q[c0:c1])
        for i in range(c0, c1):
            if i in qpos:
                bq[qpos[i]] = scale * dds[i - c0] @ np.abs(k)
    return bq, bk, bv


@pytest.mark.parametrize("causal", [False, True])
def test_backward_full_size_sampled_rows(causal):
    """The backward workload bench.py times (B=4, H=16, N=8448, d=128, bf16),
    in the same launch configuration: sampled dQ, dK and dV rows of two
    (batch, head) slices -- the first and last rows, both sides of the 64-
    and 128-row block edges, the ragged last block and seeded random rows --
    against the oracle's rows of that sequence and head, element by element
    within the first-order bound above."""
    from datagen import uniform_int
    from datagen.workloads import backward, make_dout, make_inputs
    w = backward(causal)
    x = make_inputs(w)
    do = make_dout(w)
    qd, kd, vd, dod = (t.cuda() for t in (x["q"], x["k"], x["v"], do))
    o, lse = agb.attn_fwd(qd, kd, vd, causal=causal)
    dq, dk, dv = agb.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal)
    torch.cuda.synchronize()
    assert agb.get_status() == 0
    N = w.N
    rows = sorted(set([0, 1, 63, 64, 127, 128, 4095, 4096, 8191, 8192, N - 1] +
                      [int(r) for r in uniform_int(w.seed, 40, 6, 0, N - 1)]))
    u = rel_round(torch.bfloat16)
    for b, h in ((1, 5), (3, 12)):
        sl = [t[b, :, h:h + 1].float().numpy() for t in (x["q"], x["k"], x["v"], do)]
        rq, rk, rv = oracle.attention_backward_rows(*sl, w.scale, causal, 0, rows, rows, threads())
        bq, bk, bv = bounds_rows(*(t[:, 0] for t in sl), w.scale, causal, u, rows, rows)
        got = {"dq": dq[b, rows, h].float().cpu().numpy(), "dk": dk[b, rows, h].float().cpu().numpy(),
               "dv": dv[b, rows, h].float().cpu().numpy()}
        for name, ref, bnd in (("dq", rq[0], bq), ("dk", rk, bk), ("dv", rv, bv)):
            tol = bnd + half_ulp(ref, torch.bfloat16) + 1e-4 * np.abs(ref).max()
            err = np.abs(got[name] - ref)
            print(f"({b},{h}) {name}: max err {err.max():.3e}, max |ref| {np.abs(ref).max():.3e}")
            assert np.all(err <= tol), (name, b, h, float((err - tol).max()))
