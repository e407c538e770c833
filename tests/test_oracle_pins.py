"""Pins for the fp64 oracle: checks against what the pages and the mathematics
fix, independent of the oracle's own code.

Each test names the plausible mistake it would catch.  Sources: "Fused
attention kernel" (wikillm concept card) -- Overview (exact attention),
Implementation sketch (running softmax, lse), "8-bit forward pass (FP8,
Hopper)" (e4m3, block scales, sign-diagonal x Hadamard rotation).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from datagen import normal, random_signs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(seed, shape, s=0):
    return normal(seed, s, shape, dtype=np.float64)


def dense(q, k, v, scale, causal):
    return oracle.attention(q, k, v, scale, causal)


# --------------------------------------------------------------------------
# Closed forms and hand-derived fixtures
# --------------------------------------------------------------------------

def test_golden_closed_forms():
    """Hand-derived values (catches a wrong normaliser, a missing scale, a
    natural-vs-base-2 log in lse, and causal alignment)."""
    g = json.load(open(os.path.join(GOLDEN, "attention_closed_form.json")))
    for c in g["cases"]:
        q = np.array(c["q"], dtype=np.float64)[None, :, None, :]
        k = np.array(c["k"], dtype=np.float64)[None, :, None, :]
        v = np.array(c["v"], dtype=np.float64)[None, :, None, :]
        o, lse = dense(q, k, v, c["scale"], c["causal"])
        np.testing.assert_allclose(o[0, :, 0, :], np.array(c["o"]), rtol=0, atol=1e-13,
                                   err_msg=c["name"])
        np.testing.assert_allclose(lse[0, 0], np.array(c["lse"]), rtol=0, atol=1e-13,
                                   err_msg=c["name"])


@pytest.mark.parametrize("causal", [False, True])
def test_q_zero_gives_mean_of_v(causal):
    """Q = 0: every allowed key has the same score, so O_i is the mean of the
    allowed V rows and lse_i = ln(#keys)."""
    B, N, H, d = 2, 37, 3, 16
    q = np.zeros((B, N, H, d))
    k = rnd(1, (B, N, H, d), 1)
    v = rnd(1, (B, N, H, d), 2)
    o, lse = dense(q, k, v, 0.25, causal)
    for i in range(N):
        n = i + 1 if causal else N
        np.testing.assert_allclose(o[:, i], v[:, :n].mean(axis=1), atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], math.log(n), atol=1e-13)


def test_scale_zero_gives_mean_of_v():
    B, N, H, d = 1, 20, 2, 8
    q, k, v = rnd(2, (B, N, H, d), 0), rnd(2, (B, N, H, d), 1), rnd(2, (B, N, H, d), 2)
    o, lse = dense(q, k, v, 0.0, False)
    np.testing.assert_allclose(o[0], np.broadcast_to(v[0].mean(axis=0), o[0].shape), atol=1e-13)
    np.testing.assert_allclose(lse, math.log(N), atol=1e-13)


def test_dominant_key_returns_its_value():
    """One key scoring 60 above all others: O_i = v_j* to within e^-60 (catches
    a max taken over the wrong axis, or weights applied to the wrong V row)."""
    N, d = 24, 8
    q = rnd(3, (1, N, 1, d), 0)
    k = rnd(3, (1, N, 1, d), 1) * 1e-3
    v = rnd(3, (1, N, 1, d), 2)
    i, jstar = 5, 17
    qi = q[0, i, 0]
    k[0, jstar, 0] = 60.0 * qi / float(qi @ qi)        # score exactly 60 at scale 1
    o, lse = dense(q, k, v, 1.0, False)
    np.testing.assert_allclose(o[0, i, 0], v[0, jstar, 0], atol=1e-12)
    # lse = 60 + log(1 + sum of the small exps): within 1e-20 of 60 + tiny terms
    s = np.array([qi @ k[0, j, 0] for j in range(N)])
    assert abs(lse[0, 0, i] - (60.0 + math.log1p(np.exp(s - 60.0)[np.arange(N) != jstar].sum()))) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one_and_reproduce_o(causal):
    N, H, d = 19, 2, 8
    q, k, v = rnd(4, (N, H, d), 0), rnd(4, (N, H, d), 1), rnd(4, (N, H, d), 2)
    p = oracle.probs(q, k, 0.4, causal)
    np.testing.assert_allclose(p.sum(axis=-1), 1.0, atol=1e-14)
    if causal:
        assert np.all(np.triu(p, 1) == 0.0)
    o, _ = dense(q[None], k[None], v[None], 0.4, causal)
    for h in range(H):
        np.testing.assert_allclose(p[h] @ v[:, h], o[0, :, h], atol=1e-13)


def test_causal_row_zero_is_v0():
    """Causal row 0 sees only key 0: O_0 = v_0 and lse_0 = s_00 (top-left
    alignment; catches an off-by-one in the mask)."""
    B, N, H, d = 2, 9, 3, 16
    q, k, v = rnd(5, (B, N, H, d), 0), rnd(5, (B, N, H, d), 1), rnd(5, (B, N, H, d), 2)
    o, lse = dense(q, k, v, 0.3, True)
    np.testing.assert_allclose(o[:, 0], v[:, 0], atol=1e-14)
    s00 = 0.3 * np.einsum("bhc,bhc->bh", q[:, 0], k[:, 0])
    np.testing.assert_allclose(lse[:, :, 0], s00, atol=1e-13)


# --------------------------------------------------------------------------
# Library routines and an independent derivation
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 1, 4), (2, 13, 3, 16), (1, 33, 2, 64)])
def test_matches_torch_sdpa_float64(shape, causal):
    """torch.nn.functional.scaled_dot_product_attention in float64 on the CPU,
    and torch.logsumexp of the scaled scores for lse (catches a transposed
    operand, a dropped scale, a wrong mask orientation)."""
    B, N, H, d = shape
    q, k, v = rnd(6, shape, 0), rnd(6, shape, 1), rnd(6, shape, 2)
    scale = 1.0 / math.sqrt(d)
    o, lse = dense(q, k, v, scale, causal)
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                           scale=scale)
    np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), atol=1e-12)
    s = scale * (tq @ tk.transpose(-1, -2))
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


def online_softmax_block(q, keys, values, block_c, scale, nkeys_allowed):
    """The card's running-softmax loop (Implementation sketch), restated in
    numpy for one query block, with the scale and a per-row key limit added.
    Every key block is scored, including a ragged last one."""
    Br, d = q.shape
    o = np.zeros((Br, values.shape[1]))
    m = np.full(Br, -np.inf)
    l = np.zeros(Br)
    N = keys.shape[0]
    for j in range(-(-N // block_c)):
        kb = keys[j * block_c:(j + 1) * block_c]
        vb = values[j * block_c:(j + 1) * block_c]
        s = scale * (q @ kb.T)
        cols = np.arange(j * block_c, j * block_c + kb.shape[0])
        s = np.where(cols[None, :] < nkeys_allowed[:, None], s, -np.inf)
        m_new = np.maximum(m, s.max(axis=1))
        alpha = np.where(np.isneginf(m_new), 1.0, np.exp(m - m_new))
        p = np.where(np.isneginf(s), 0.0, np.exp(s - m_new[:, None]))
        l = alpha * l + p.sum(axis=1)
        o = alpha[:, None] * o + p @ vb
        m = m_new
    return o / l[:, None], m + np.log(l)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,block_c", [(10, 3), (16, 4), (7, 16)])
def test_matches_running_softmax_loop(N, block_c, causal):
    """The plain two-pass definition and the card's blockwise running-softmax
    loop must agree to rounding (catches an inverted rescale factor or a
    skipped last key block -- the two errata the card reports)."""
    H, d = 2, 8
    q, k, v = rnd(7, (N, H, d), 0), rnd(7, (N, H, d), 1), rnd(7, (N, H, d), 2)
    o, lse = dense(q[None], k[None], v[None], 0.37, causal)
    allowed = (np.arange(N) + 1) if causal else np.full(N, N)
    for h in range(H):
        oo, ll = online_softmax_block(q[:, h], k[:, h], v[:, h], block_c, 0.37, allowed)
        np.testing.assert_allclose(o[0, :, h], oo, atol=1e-12)
        np.testing.assert_allclose(lse[0, h], ll, atol=1e-12)


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------

def test_key_permutation_invariance():
    B, N, H, d = 1, 23, 2, 16
    q, k, v = rnd(8, (B, N, H, d), 0), rnd(8, (B, N, H, d), 1), rnd(8, (B, N, H, d), 2)
    perm = np.random.default_rng(0).permutation(N)
    o1, l1 = dense(q, k, v, 0.25, False)
    o2, l2 = dense(q, k[:, perm], v[:, perm], 0.25, False)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_key_shift_shifts_lse_only():
    """k_j -> k_j + c for every key: lse_i shifts by scale*q_i.c, O unchanged."""
    B, N, H, d = 1, 17, 2, 8
    q, k, v = rnd(9, (B, N, H, d), 0), rnd(9, (B, N, H, d), 1), rnd(9, (B, N, H, d), 2)
    c = rnd(9, (d,), 3)
    o1, l1 = dense(q, k, v, 0.5, True)
    o2, l2 = dense(q, k + c, v, 0.5, True)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    shift = 0.5 * np.einsum("bnhc,c->bhn", q, c)
    np.testing.assert_allclose(l2 - l1, shift, atol=1e-12)


def test_varlen_sequence_equals_dense_call():
    H, d = 2, 16
    lens = [5, 1, 12, 7]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v = rnd(10, (T, H, d), 0), rnd(10, (T, H, d), 1), rnd(10, (T, H, d), 2)
    for causal in (False, True):
        o, lse = oracle.attention_varlen(q, k, v, cu, 0.3, causal)
        for s, L in enumerate(lens):
            a, b = cu[s], cu[s + 1]
            od, ld = dense(q[None, a:b], k[None, a:b], v[None, a:b], 0.3, causal)
            np.testing.assert_allclose(o[a:b], od[0], atol=1e-14)
            np.testing.assert_allclose(lse[:, a:b], ld[0], atol=1e-14)


def test_row_subset_equals_full():
    B, N, H, d = 2, 31, 3, 8
    q, k, v = rnd(11, (B, N, H, d), 0), rnd(11, (B, N, H, d), 1), rnd(11, (B, N, H, d), 2)
    o, lse = dense(q, k, v, 0.35, True)
    tok = np.array([0, 30, 31, 45, 61])
    head = np.array([2, 0, 1, 2, 0])
    cu = (np.arange(B + 1) * N).astype(np.int32)
    ro, rl = oracle.attention_rows(q.reshape(B * N, H, d), k.reshape(B * N, H, d),
                                   v.reshape(B * N, H, d), cu, 0.35, True, tok, head)
    for r, (t, h) in enumerate(zip(tok, head)):
        np.testing.assert_array_equal(ro[r], o[t // N, t % N, h])
        assert rl[r] == lse[t // N, h, t % N]


def test_rejects_bad_arguments():
    q = np.zeros((4, 1, 8))
    with pytest.raises(ValueError):
        oracle.attention_rows(q, q, q, np.array([0, 3, 2], dtype=np.int32), 1.0, False,
                              [0], [0])
    with pytest.raises(ValueError):
        oracle.attention_rows(q, q, q, np.array([0, 4], dtype=np.int32), 1.0, False,
                              [0], [1])
    with pytest.raises(ValueError):
        oracle.hadamard_matrix(12)


# --------------------------------------------------------------------------
# Incoherent processing (sign diagonal x Hadamard)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("d", [1, 2, 8, 64, 128])
def test_hadamard_is_sylvester(d):
    """The Hadamard matrix is Sylvester's construction (scipy.linalg.hadamard)."""
    scipy_linalg = pytest.importorskip("scipy.linalg")
    np.testing.assert_array_equal(oracle.hadamard_matrix(d), scipy_linalg.hadamard(d))


@pytest.mark.parametrize("d", [64, 128])
def test_rotation_is_orthogonal(d):
    """M = diag(s) H / sqrt(d): rows of I*M are M's rows; M M^T = I and norms
    are preserved (catches a missing 1/sqrt(d) or a sign applied twice)."""
    s = random_signs(77, d)
    m = oracle.rotate(np.eye(d), s)
    np.testing.assert_allclose(m @ m.T, np.eye(d), atol=1e-14)
    expect = np.diag(s.astype(np.float64)) @ oracle.hadamard_matrix(d) / math.sqrt(d)
    np.testing.assert_allclose(m, expect, atol=1e-15)
    x = rnd(12, (50, d))
    np.testing.assert_allclose(np.linalg.norm(oracle.rotate(x, s), axis=1),
                               np.linalg.norm(x, axis=1), rtol=1e-14)


def test_rotation_leaves_attention_unchanged():
    """The orthogonal matrix cancels in Q K^T, so attention on (QM, KM, V)
    equals attention on (Q, K, V)."""
    B, N, H, d = 1, 40, 2, 64
    q, k, v = rnd(13, (B, N, H, d), 0), rnd(13, (B, N, H, d), 1), rnd(13, (B, N, H, d), 2)
    s = random_signs(13, d)
    o1, l1 = dense(q, k, v, 0.125, False)
    o2, l2 = dense(oracle.rotate(q, s), oracle.rotate(k, s), v, 0.125, False)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)
    # a rotation applied to Q only does change the result
    o3, _ = dense(oracle.rotate(q, s), k, v, 0.125, False)
    assert np.abs(o3 - o1).max() > 1e-2


# --------------------------------------------------------------------------
# e4m3 and block quantisation
# --------------------------------------------------------------------------

def test_e4m3_fixture_codes():
    g = json.load(open(os.path.join(GOLDEN, "e4m3_codes.json")))
    for code, val in g["decode"]:
        got = oracle.e4m3_decode(np.array([int(code, 16)], dtype=np.uint8))[0]
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code
    for val, code in g["encode_rne_satfinite"]:
        assert oracle.e4m3_encode(np.array([val]))[0] == int(code, 16), val


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    np.testing.assert_array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])


def test_e4m3_encode_matches_torch_in_range():
    """Round-to-nearest-even against torch's float64 -> float8_e4m3fn cast,
    on random values, all exact values and all midpoints within +-448."""
    vals = oracle.e4m3_decode(np.arange(0, 127, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    x = np.concatenate([vals, mids, -vals, -mids,
                        rnd(14, (20000,)) * 30, rnd(14, (2000,), 1) * 1e-3])
    x = x[np.abs(x) <= 448]
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    zero = (oracle.e4m3_decode(ours) == 0)
    np.testing.assert_array_equal(ours[~zero], ref[~zero])
    np.testing.assert_array_equal(oracle.e4m3_decode(ref[zero]), 0.0)


def test_e4m3_saturates():
    c = oracle.e4m3_encode(np.array([448.0, 470.0, 1e30, -1e30, np.inf]))
    np.testing.assert_array_equal(c, [0x7E, 0x7E, 0x7E, 0xFE, 0x7E])


@pytest.mark.parametrize("per_tensor", [False, True])
def test_block_quant_scales_and_error_bound(per_tensor):
    """scale = amax/448: the block's largest entry maps to +-448 exactly, every
    entry is within half an e4m3 step (at its magnitude) of its true value."""
    B, N, H, d = 2, 300, 2, 16
    x = rnd(15, (B, N, H, d)) * np.exp(rnd(15, (B, N, H, 1), 1))
    codes, desc = oracle.block_quant(x, per_tensor)
    nblk = -(-N // 128)
    assert desc.shape == (B, H, nblk)
    for b in range(B):
        for h in range(H):
            for j in range(nblk):
                blk = x[b, j * 128:(j + 1) * 128, h]
                amax = np.abs(x).max() if per_tensor else np.abs(blk).max()
                assert desc[b, h, j] == amax / 448.0
    deq = oracle.dequantize(codes, desc)
    scl = desc[:, :, np.arange(N) // 128].transpose(0, 2, 1)[..., None]
    y = np.abs(x) / scl                                     # magnitude in code units
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    half_step = 2.0 ** (e - 3) / 2                          # 3 mantissa bits
    assert np.all(np.abs(deq - x) <= half_step * scl * (1 + 1e-12))
    # the largest entry of each block lands exactly on 448
    assert np.max(np.abs(oracle.e4m3_decode(codes))) == 448.0


def test_zero_block_gets_scale_one():
    x = np.zeros((1, 130, 1, 8))
    x[0, 129, 0, 3] = 2.0
    codes, desc = oracle.block_quant(x)
    assert desc[0, 0, 0] == 1.0 and desc[0, 0, 1] == 2.0 / 448.0
    assert np.all(codes[0, :128] == 0)
    assert oracle.e4m3_decode(codes[0, 129, 0, 3:4])[0] == 448.0


def test_quantize_qkv_rotates_q_and_k_only():
    B, N, H, d = 1, 128, 1, 64
    q, k, v = rnd(16, (B, N, H, d), 0), rnd(16, (B, N, H, d), 1), rnd(16, (B, N, H, d), 2)
    s = random_signs(16, d)
    r = oracle.quantize_qkv(q, k, v, s)
    np.testing.assert_allclose(r["q_rot"], oracle.rotate(q, s))
    np.testing.assert_allclose(oracle.dequantize(r["v8"], r["dv"]), v, atol=np.abs(v).max() / 448 * 16)
    # dequantised q.k matches the unrotated q.k to fp8 accuracy
    qd, kd = oracle.dequantize(r["q8"], r["dq"]), oracle.dequantize(r["k8"], r["dk"])
    s_ref = np.einsum("nc,mc->nm", q[0, :, 0], k[0, :, 0])
    s_q = np.einsum("nc,mc->nm", qd[0, :, 0], kd[0, :, 0])
    assert np.sqrt(np.mean((s_q - s_ref) ** 2)) < 0.1 * np.sqrt(np.mean(s_ref ** 2))


# --------------------------------------------------------------------------
# Inference variants: grouped K/V heads, queries at the end of the keys,
# paged keys, and the merge of partial results over key ranges
# (HippoAttention case study, "Our approach": paged attention;
# FlashAttention-3 summary, Limitations: LLM inference)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("hkv", [1, 2, 4])
def test_gqa_matches_torch_sdpa_float64(hkv, causal):
    """Grouped K/V heads against torch's own grouped-query SDPA in float64
    (catches a wrong head mapping, e.g. h % Hkv instead of h // (H/Hkv))."""
    B, N, H, d = 2, 19, 8, 16
    q, k, v = rnd(50, (B, N, H, d)), rnd(50, (B, N, hkv, d), 1), rnd(50, (B, N, hkv, d), 2)
    o, lse = oracle.attention_gqa(q, k, v, 0.3, causal)
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                           scale=0.3, enable_gqa=True)
    np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)
    # lse against an explicit log-sum-exp over the grouped heads' scores
    kr = np.repeat(k, H // hkv, axis=2)
    s = np.einsum("bnhd,bmhd->bhnm", q, kr) * 0.3
    if causal:
        s = np.where(np.tril(np.ones((N, N), bool)), s, -np.inf)
    np.testing.assert_allclose(lse, np.logaddexp.reduce(s, axis=3), rtol=0, atol=1e-12)


def test_gqa_equals_attention_with_repeated_kv_heads():
    """Grouping reduces to plain attention on K/V heads repeated per group."""
    B, N, H, hkv, d = 2, 23, 6, 3, 8
    q, k, v = rnd(51, (B, N, H, d)), rnd(51, (B, N, hkv, d), 1), rnd(51, (B, N, hkv, d), 2)
    for causal in (False, True):
        o, lse = oracle.attention_gqa(q, k, v, 0.4, causal)
        o2, lse2 = oracle.attention(q, np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2), 0.4,
                                    causal)
        np.testing.assert_array_equal(o, o2)
        np.testing.assert_array_equal(lse, lse2)


def test_queries_at_the_end_equal_the_last_rows_of_full_causal_attention():
    """Nq queries against Nk >= Nq keys, causal: they are the last Nq
    positions, so the result equals the last Nq rows of square causal
    attention (catches top-left alignment where the keys are longer)."""
    B, Nk, Nq, H, d = 2, 40, 7, 2, 8
    qf, k, v = rnd(52, (B, Nk, H, d)), rnd(52, (B, Nk, H, d), 1), rnd(52, (B, Nk, H, d), 2)
    of, lf = oracle.attention(qf, k, v, 0.5, True)
    o, lse = oracle.attention_gqa(qf[:, Nk - Nq:], k, v, 0.5, True)
    np.testing.assert_array_equal(o, of[:, Nk - Nq:])
    np.testing.assert_array_equal(lse, lf[:, :, Nk - Nq:])


def test_queries_at_the_end_match_torch_with_explicit_mask():
    B, Nk, Nq, H, d = 1, 11, 4, 2, 8
    q, k, v = rnd(53, (B, Nq, H, d)), rnd(53, (B, Nk, H, d), 1), rnd(53, (B, Nk, H, d), 2)
    o, _ = oracle.attention_gqa(q, k, v, 0.5, True)
    mask = torch.from_numpy(np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq))
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask,
                                                           scale=0.5)
    np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)


def test_query_with_no_allowed_key_is_empty():
    """More queries than keys, causal: the first Nq - Nk queries see no key
    (O = 0, lse = -inf by the stated convention)."""
    q, k, v = rnd(54, (1, 5, 1, 4)), rnd(54, (1, 3, 1, 4), 1), rnd(54, (1, 3, 1, 4), 2)
    o, lse = oracle.attention_gqa(q, k, v, 1.0, True)
    assert np.all(o[0, :2] == 0) and np.all(np.isneginf(lse[0, 0, :2]))
    assert np.isfinite(lse[0, 0, 2:]).all()


@pytest.mark.parametrize("causal", [False, True])
def test_paged_equals_contiguous(causal):
    """Keys read through a shuffled page table give the contiguous result
    (catches a wrong page / row split of the token index)."""
    B, H, hkv, d, P = 3, 4, 2, 8, 16
    seqlens = [37, 16, 50]
    Nq = 5
    npages = sum((L + P - 1) // P for L in seqlens) + 3
    rng = np.random.default_rng(55)
    perm = rng.permutation(npages)
    kc, vc = rnd(55, (npages, P, hkv, d), 1), rnd(55, (npages, P, hkv, d), 2)
    table, used = [], 0
    for L in seqlens:
        n = (L + P - 1) // P
        table.append(perm[used:used + n])
        used += n
    q = rnd(55, (B, Nq, H, d))
    o, lse = oracle.attention_paged(q, kc, vc, table, seqlens, 0.35, causal)
    for b, L in enumerate(seqlens):
        rows = np.concatenate([np.arange(P) + P * pg for pg in table[b]])[:L]
        kb = kc.reshape(-1, hkv, d)[rows][None]
        vb = vc.reshape(-1, hkv, d)[rows][None]
        ob, lb = oracle.attention_gqa(q[b:b + 1], kb, vb, 0.35, causal)
        np.testing.assert_array_equal(o[b], ob[0])
        np.testing.assert_array_equal(lse[b], lb[0])


def test_merge_of_key_ranges_equals_unsplit_attention():
    """Attention over disjoint key ranges, merged, equals attention over all
    keys (the combine step of split-key decoding), including an empty part."""
    N, H, d = 45, 2, 8
    q, k, v = rnd(56, (1, N, H, d)), rnd(56, (1, N, H, d), 1), rnd(56, (1, N, H, d), 2)
    o_full, lse_full = oracle.attention_gqa(q[:, :3], k, v, 0.4, False)
    bounds = [0, 10, 10, 31, 45]                       # the second part is empty
    parts_o, parts_l = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b > a:
            o_s, l_s = oracle.attention_gqa(q[:, :3], k[:, a:b], v[:, a:b], 0.4, False)
        else:
            o_s, l_s = np.zeros((1, 3, H, d)), np.full((1, H, 3), -np.inf)
        parts_o.append(o_s[0].reshape(3 * H, d))
        parts_l.append(l_s[0].T.reshape(3 * H))
    o, lse = oracle.merge_partials(np.stack(parts_o), np.stack(parts_l))
    np.testing.assert_allclose(o, o_full[0].reshape(3 * H, d), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_full[0].T.reshape(3 * H), rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# Additive score bias ("[+mask]" of the problem statement; "Bias" among the
# additions of the HippoAttention case study, "Our approach")
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_bias_matches_torch_sdpa_float64(causal):
    """A per-(batch, head, query, key) bias against torch's SDPA with the same
    float mask in float64 (catches a transposed bias or a wrong stride)."""
    B, N, H, d = 2, 13, 3, 8
    q, k, v = rnd(60, (B, N, H, d)), rnd(60, (B, N, H, d), 1), rnd(60, (B, N, H, d), 2)
    bias = 2.0 * rnd(60, (B, H, N, N), 3)
    o, lse = oracle.attention_bias(q, k, v, bias, 0.35, causal)
    mask = torch.from_numpy(bias.copy())
    if causal:
        mask = mask.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=0.35)
    np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)
    s = np.einsum("bnhd,bmhd->bhnm", q, k) * 0.35 + mask.numpy()
    np.testing.assert_allclose(lse, np.logaddexp.reduce(s, axis=3), rtol=0, atol=1e-12)


def test_constant_bias_shifts_lse_only():
    B, N, H, d = 1, 17, 2, 8
    q, k, v = rnd(61, (B, N, H, d)), rnd(61, (B, N, H, d), 1), rnd(61, (B, N, H, d), 2)
    o0, l0 = oracle.attention(q, k, v, 0.5, True)
    o1, l1 = oracle.attention_bias(q, k, v, np.full((1, 1, 1, N), 3.25), 0.5, True)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1, l0 + 3.25, rtol=0, atol=1e-13)


def test_minus_inf_bias_removes_keys():
    """A key-mask bias (0 or -inf per key, broadcast over heads and queries)
    equals attention over the kept keys only; a row with every key removed is
    empty."""
    B, N, H, d = 2, 20, 2, 8
    q, k, v = rnd(62, (B, N, H, d)), rnd(62, (B, N, H, d), 1), rnd(62, (B, N, H, d), 2)
    keep = np.ones((B, N), bool)
    keep[0, [1, 5, 6, 19]] = False
    keep[1, 10:] = False
    bias = np.where(keep, 0.0, -np.inf)[:, None, None, :]
    o, lse = oracle.attention_bias(q, k, v, bias, 0.4, False)
    for b in range(B):
        ob, lb = oracle.attention_gqa(q[b:b + 1], k[b:b + 1, keep[b]], v[b:b + 1, keep[b]], 0.4,
                                      False)
        np.testing.assert_allclose(o[b], ob[0], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[b], lb[0], rtol=0, atol=1e-13)
    o2, l2 = oracle.attention_bias(q, k, v, np.full((1, 1, 1, N), -np.inf), 0.4, False)
    assert np.all(o2 == 0) and np.all(np.isneginf(l2))


# --------------------------------------------------------------------------
# Backward pass (FlashAttention-3 summary, Key Results; the card's "When to
# use which": backward pass needed)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("hkv", [1, 2, 4])
def test_backward_matches_torch_autograd_float64(hkv, causal):
    """dQ, dK, dV against torch autograd through float64 SDPA (catches a
    missing softmax-Jacobian term, a dropped scale, dK/dV not summed over a
    group's query heads, or gradients leaking through masked keys)."""
    B, N, H, d = 2, 11, 4, 8
    q, k, v = rnd(70, (B, N, H, d)), rnd(70, (B, N, hkv, d), 1), rnd(70, (B, N, hkv, d), 2)
    do = rnd(70, (B, N, H, d), 3)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.3, causal)
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3).requires_grad_() for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=0.3,
                                                         enable_gqa=True)
    o.backward(torch.from_numpy(do).permute(0, 2, 1, 3))
    for mine, t in ((dq, tq), (dk, tk), (dv, tv)):
        np.testing.assert_allclose(mine, t.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)


def test_backward_matches_finite_differences_of_the_forward():
    """Central differences of sum(dO * O) through the oracle's own forward."""
    B, N, H, d = 1, 6, 1, 4
    q, k, v, do = (rnd(71, (B, N, H, d), s) for s in range(4))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.7, True)
    def f(q_, k_, v_):
        return float((oracle.attention(q_, k_, v_, 0.7, True)[0] * do).sum())
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        for idx in [(0, 0, 0, 0), (0, 3, 0, 2), (0, 5, 0, 3), (0, 2, 0, 1)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if y is x else y for y in (q, k, v)]
            args_m = [xm if y is x else y for y in (q, k, v)]
            num = (f(*args_p) - f(*args_m)) / (2 * eps)
            assert abs(num - g[idx]) < 1e-7, (idx, num, g[idx])


def test_backward_dv_sums_to_do_and_single_key_rows_have_no_dq():
    """Rows of P sum to 1, so sum_j dV_j = sum_i dO_i; the first causal row
    has one key, so its softmax is constant and dQ there is 0."""
    B, N, H, d = 2, 9, 3, 8
    q, k, v, do = (rnd(72, (B, N, H, d), s) for s in range(4))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.5, True)
    np.testing.assert_allclose(dv.sum(axis=1), do.sum(axis=1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq[:, 0], 0.0, rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_rows_match_torch_autograd_float64(causal):
    """Selected rows of one sequence's gradients (the form the full-size GPU
    checks use) against torch autograd through float64 SDPA: every query
    head of the chosen K/V head's group for dQ, the group sum for dK, dV."""
    L, H, hkv, d = 37, 6, 2, 8
    q, do = rnd(73, (1, L, H, d)), rnd(73, (1, L, H, d), 3)
    k, v = rnd(73, (1, L, hkv, d), 1), rnd(73, (1, L, hkv, d), 2)
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3).requires_grad_() for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=0.45,
                                                         enable_gqa=True)
    o.backward(torch.from_numpy(do).permute(0, 2, 1, 3))
    gq, gk, gv = (t.grad.permute(0, 2, 1, 3).numpy()[0] for t in (tq, tk, tv))
    qrows, krows = [0, 1, 17, 36], [0, 5, 35, 36]
    g = H // hkv
    for hk in range(hkv):
        dq, dk, dv = oracle.attention_backward_rows(q[0], k[0], v[0], do[0], 0.45, causal, hk,
                                                    qrows, krows, nthreads=3)
        for gh in range(g):
            np.testing.assert_allclose(dq[gh], gq[qrows, hk * g + gh], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk, gk[krows, hk], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv, gv[krows, hk], rtol=0, atol=1e-12)


def test_backward_rows_agree_with_the_full_backward():
    """The rows entry point and the full backward on the same sequence."""
    L, H, hkv, d = 50, 4, 1, 16
    q, k, v, do = (rnd(74, (1, L, h, d), s) for s, h in enumerate((H, hkv, hkv, H)))
    fq, fk, fv = oracle.attention_backward(q, k, v, do, 0.25, True)
    rows = list(range(0, L, 7)) + [L - 1]
    dq, dk, dv = oracle.attention_backward_rows(q[0], k[0], v[0], do[0], 0.25, True, 0, rows,
                                                rows)
    np.testing.assert_allclose(dq, fq[0][rows].transpose(1, 0, 2), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk, fk[0][rows, 0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, fv[0][rows, 0], rtol=0, atol=1e-13)
