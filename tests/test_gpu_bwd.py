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
value for fp32 accumulation order (atomic dQ sums) and the exp2
approximation.  |P|, |dS| for the bound are formed in float64 here; the
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
@pytest.mark.parametrize("N,H,Hkv", [(128, 2, 2), (300, 4, 2), (513, 3, 1)])
def test_backward_parity(N, H, Hkv, causal, dtype):
    B, d = 2, 128
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
