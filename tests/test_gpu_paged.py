"""GPU parity of decoding against a paged K/V cache (attn_fwd_paged) with
the fp64 oracle, element by element: grouped K/V heads, several page sizes,
ragged and empty sequences, causal (queries at the end of the keys) and not,
one split or many (the split results merged); plus exactness of the page
indirection: pages the table does not name are never read."""
import math

import numpy as np
import pytest
import torch

import attention_forward_softmax_gb300 as agb
import oracle
from datagen import normal, to_bf16, to_fp16, uniform_int
from tests._gpu_helpers import TOL_LSE, assert_close_o, n_eff, threads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    agb.build()
    agb.lib()


def make_cache(seed, seqlens, page_size, Hkv, d, dtype, spare=3):
    """A cache whose pages are handed out in a seeded random order."""
    conv = to_bf16 if dtype == torch.bfloat16 else to_fp16
    need = [(L + page_size - 1) // page_size for L in seqlens]
    npages = sum(need) + spare
    perm = np.argsort(uniform_int(seed, 20, npages, 0, 1 << 30), kind="stable")
    maxp = max(1, max(need))
    table = np.zeros((len(seqlens), maxp), dtype=np.int32)
    used = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[used:used + n]
        used += n
    kc = conv(normal(seed, 21, (npages, page_size, Hkv, d)))
    vc = conv(normal(seed, 22, (npages, page_size, Hkv, d)))
    return kc, vc, table, perm[used:]


def check(seed, seqlens, Nq, H, Hkv, d, page_size, causal, splits, dtype=torch.bfloat16):
    conv = to_bf16 if dtype == torch.bfloat16 else to_fp16
    B = len(seqlens)
    kc, vc, table, _ = make_cache(seed, seqlens, page_size, Hkv, d, dtype)
    q = conv(normal(seed, 23, (B, Nq, H, d)))
    scale = 1 / math.sqrt(d)
    o, lse = agb.attn_fwd_paged(q.cuda(), kc.cuda(), vc.cuda(), torch.from_numpy(table).cuda(),
                                torch.tensor(seqlens, dtype=torch.int32).cuda(),
                                max(1, max(seqlens)), causal=causal, num_splits=splits)
    torch.cuda.synchronize()
    assert agb.get_status() == 0
    o_ref, lse_ref = oracle.attention_paged(q, kc, vc, table, seqlens, scale, causal, threads())
    a_ref, _ = oracle.attention_paged(q, kc, vc.abs(), table, seqlens, scale, causal, threads())
    _, lse2 = oracle.attention_paged(q, kc, vc, table, seqlens, 2 * scale, causal, threads())
    og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
    empty = np.isneginf(lse_ref)
    ne = n_eff(np.where(empty, 0, lse_ref), np.where(empty, 0, lse2)).transpose(0, 2, 1)[..., None]
    assert_close_o(og, o_ref, a_ref, dtype, ne, f"paged {seqlens} Nq={Nq} splits={splits}")
    assert np.array_equal(np.isneginf(lg), empty)
    assert np.all(og[empty.transpose(0, 2, 1)] == 0)
    if (~empty).any():
        assert np.abs(lg[~empty] - lse_ref[~empty]).max() <= TOL_LSE
    return og, lg


@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_paged_decode_parity(d, causal, splits):
    check(6000 + d, [1, 300, 777, 129, 2048], 1, 8, 2, d, 16, causal, splits)


@pytest.mark.parametrize("page_size", [1, 7, 16, 48, 64, 96, 256])
def test_paged_page_sizes(page_size):
    check(6100 + page_size, [513, 64, 1000], 2, 4, 1, 128, page_size, True, 0)


@pytest.mark.parametrize("Nq,H,Hkv", [(4, 4, 1), (2, 8, 1), (16, 1, 1), (1, 16, 16)])
def test_paged_row_shapes(Nq, H, Hkv):
    check(6200 + Nq * H, [255, 1500], Nq, H, Hkv, 128, 32, True, 0)


def test_paged_fp16_and_empty_or_short_sequences():
    # a sequence without keys, and one shorter than the number of queries
    check(6300, [0, 3, 400], 4, 4, 2, 64, 16, True, 2, torch.float16)


def test_paged_unlisted_pages_are_never_read():
    seqlens = [300, 45, 1030]
    kc, vc, table, spare = make_cache(6400, seqlens, 16, 2, 128, torch.bfloat16)
    q = to_bf16(normal(6400, 23, (3, 2, 8, 128)))
    args = (torch.from_numpy(table).cuda(), torch.tensor(seqlens, dtype=torch.int32).cuda(), 1030)
    o1, l1 = agb.attn_fwd_paged(q.cuda(), kc.cuda(), vc.cuda(), *args, num_splits=4)
    kp, vp = kc.clone(), vc.clone()
    kp[spare] = float("nan")
    vp[spare] = 3e4
    # rows past each sequence's end in its last page
    for b, L in enumerate(seqlens):
        if L % 16:
            kp[table[b, L // 16], L % 16:] = float("nan")
            vp[table[b, L // 16], L % 16:] = 3e4
    o2, l2 = agb.attn_fwd_paged(q.cuda(), kp.cuda(), vp.cuda(), *args, num_splits=4)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_paged_rejects_too_many_rows_per_kv_head():
    q = torch.zeros((1, 4, 8, 64), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((2, 16, 1, 64), dtype=torch.bfloat16, device="cuda")
    t = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(agb.AttnError):
        agb.attn_fwd_paged(q, kc, kc, t, torch.tensor([20], dtype=torch.int32, device="cuda"), 20)
