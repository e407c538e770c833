"""GPU parity of grouped K/V heads (grouped-query attention; H_kv = 1 is
multi-query attention) against the fp64 oracle, element by element, dense
and packed, with ragged tails; and exactness of the head mapping: poisoning
every K/V head but a group's own leaves that group's outputs bitwise
unchanged."""
import math

import numpy as np
import pytest
import torch

import attention_forward_softmax_gb300 as agb
import oracle
from tests._gpu_helpers import (TOL_LSE, assert_close_lse, assert_close_o, n_eff, qkv,
                                threads)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    agb.build()
    agb.lib()


def oracle_gqa(q, k, v, scale, causal):
    o, lse = oracle.attention_gqa(q, k, v, scale, causal, nthreads=threads())
    a, _ = oracle.attention_gqa(q, k, v.abs(), scale, causal, nthreads=threads())
    _, lse2 = oracle.attention_gqa(q, k, v, 2 * scale, causal, nthreads=threads())
    return o, lse, a, n_eff(lse, lse2).transpose(0, 2, 1)[..., None]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv", [(8, 2), (6, 1), (4, 4)])
def test_gqa_dense_parity(H, Hkv, causal, d, dtype):
    B, N = 2, 300
    q, _, _ = qkv(5000 + H + Hkv + d, (B, N, H, d), dtype)
    _, k, v = qkv(5100 + H + Hkv + d, (B, N, Hkv, d), dtype)
    o, lse = agb.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert agb.get_status() == 0
    o_ref, lse_ref, a_ref, ne = oracle_gqa(q, k, v, 1 / math.sqrt(d), causal)
    assert_close_o(o.float().cpu().numpy(), o_ref, a_ref, dtype, ne, f"H={H} Hkv={Hkv}")
    assert_close_lse(lse.cpu().numpy(), lse_ref, "gqa")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_gqa_varlen_parity(causal, d):
    H, Hkv = 8, 2
    lens = [1, 130, 77, 256, 513, 3]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, _, _ = qkv(5200 + d, (T, H, d), torch.bfloat16)
    _, k, v = qkv(5300 + d, (T, Hkv, d), torch.bfloat16)
    o, lse = agb.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cu).cuda(),
                                 max(lens), causal=causal)
    torch.cuda.synchronize()
    assert agb.get_status() == 0
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle.attention_varlen_gqa(q, k, v, cu, cu, scale, causal, threads())
    a_ref, _ = oracle.attention_varlen_gqa(q, k, v.abs(), cu, cu, scale, causal, threads())
    _, lse2 = oracle.attention_varlen_gqa(q, k, v, cu, cu, 2 * scale, causal, threads())
    assert_close_o(o.float().cpu().numpy(), o_ref, a_ref, torch.bfloat16,
                   n_eff(lse_ref, lse2).T[..., None], "varlen gqa")
    assert_close_lse(lse.cpu().numpy(), lse_ref, "varlen gqa")


def test_gqa_other_kv_heads_are_never_read():
    """Poison every K/V head except head g: query heads of group g give
    bitwise the same output."""
    B, N, H, Hkv, d = 1, 260, 8, 4, 128
    q, _, _ = qkv(5400, (B, N, H, d), torch.bfloat16)
    _, k, v = qkv(5500, (B, N, Hkv, d), torch.bfloat16)
    o1, l1 = agb.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    g = 2
    kp, vp = k.clone(), v.clone()
    for hk in range(Hkv):
        if hk != g:
            kp[:, :, hk] = float("nan")
            vp[:, :, hk] = 3e4
    o2, l2 = agb.attn_fwd(q.cuda(), kp.cuda(), vp.cuda(), causal=True)
    torch.cuda.synchronize()
    hs = slice(g * (H // Hkv), (g + 1) * (H // Hkv))
    assert torch.equal(o1[:, :, hs].view(torch.int16), o2[:, :, hs].view(torch.int16))
    assert torch.equal(l1[:, hs].view(torch.int32), l2[:, hs].view(torch.int32))


def test_gqa_rejects_indivisible_heads():
    q = torch.zeros((1, 16, 6, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 16, 4, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(agb.AttnError):
        agb.attn_fwd(q, k, k)
