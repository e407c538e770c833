"""GPU parity of attention with an additive score bias (attn_fwd_bias)
against the fp64 oracle, element by element: full, per-head and broadcast
biases, large ALiBi-style distances, key masks of -inf, rows left with no
key, ragged tails, causal and not, both 16-bit types and head sizes."""
import math

import numpy as np
import pytest
import torch

import attention_forward_softmax_gb300 as agb
import oracle
from datagen import normal
from tests._gpu_helpers import TOL_LSE, assert_close_o, n_eff, qkv, threads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    agb.build()
    agb.lib()


def padded(bias):
    """The bias on the device with its key axis padded to a multiple of 4
    (every row then starts on a 16-byte boundary, as the call requires), as
    a view of the first N keys."""
    n = bias.shape[-1]
    buf = np.zeros(bias.shape[:-1] + ((n + 3) // 4 * 4,), np.float32)
    buf[..., :n] = bias
    return torch.from_numpy(buf).cuda()[..., :n]


def run(q, k, v, bias, causal, dtype):
    d = q.shape[-1]
    scale = 1 / math.sqrt(d)
    o, lse = agb.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, bias=padded(bias))
    torch.cuda.synchronize()
    assert agb.get_status() == 0
    b64 = bias.astype(np.float64)
    o_ref, lse_ref = oracle.attention_bias(q, k, v, b64, scale, causal, threads())
    a_ref, _ = oracle.attention_bias(q, k, v.abs(), b64, scale, causal, threads())
    _, lse2 = oracle.attention_bias(q, k, v, 2 * b64, 2 * scale, causal, threads())
    empty = np.isneginf(lse_ref)
    ne = n_eff(np.where(empty, 0, lse_ref), np.where(empty, 0, lse2)).transpose(0, 2, 1)[..., None]
    og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
    assert_close_o(og, o_ref, a_ref, dtype, ne, "bias")
    assert np.array_equal(np.isneginf(lg), empty)
    if (~empty).any():
        assert np.abs(lg[~empty] - lse_ref[~empty]).max() <= TOL_LSE
    assert np.all(og.transpose(0, 2, 1, 3)[empty] == 0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_full_bias(causal, d, dtype):
    B, N, H = 2, 300, 3
    q, k, v = qkv(7000 + d, (B, N, H, d), dtype)
    bias = 2.0 * normal(7000 + d, 5, (B, H, N, N))
    run(q, k, v, bias, causal, dtype)


@pytest.mark.parametrize("causal", [False, True])
def test_alibi_distances_per_head(causal):
    """Per-head linear distance penalties with magnitudes in the thousands
    (fp32 keeps them exact enough), broadcast over the batch."""
    B, N, H, d = 2, 1100, 4, 128
    q, k, v = qkv(7100, (B, N, H, d), torch.bfloat16)
    slopes = 2.0 ** (-np.arange(1, H + 1))
    dist = np.abs(np.arange(N)[:, None] - np.arange(N)[None, :])
    bias = (-slopes[:, None, None] * dist[None])[None]           # [1, H, N, N]
    run(q, k, v, bias, causal, torch.bfloat16)


def test_key_mask_and_rows_without_keys():
    """A [B, 1, 1, N] key mask of 0 / -inf, with one batch entry's keys all
    removed (its rows come out empty)."""
    B, N, H, d = 3, 257, 2, 64
    q, k, v = qkv(7200, (B, N, H, d), torch.bfloat16)
    keep = np.ones((B, N), bool)
    keep[0, ::3] = False
    keep[1, 100:] = False
    keep[2, :] = False
    bias = np.where(keep, 0.0, -np.inf)[:, None, None, :]
    run(q, k, v, bias, False, torch.bfloat16)


def test_bias_with_grouped_heads():
    B, N, H, Hkv, d = 1, 260, 8, 2, 128
    q, _, _ = qkv(7300, (B, N, H, d), torch.bfloat16)
    _, k, v = qkv(7301, (B, N, Hkv, d), torch.bfloat16)
    bias = normal(7300, 5, (1, H, N, N))
    run(q, k, v, bias, True, torch.bfloat16)


def test_bias_rejects_misaligned_strides():
    q = torch.zeros((1, 16, 2, 64), dtype=torch.bfloat16, device="cuda")
    bias = torch.zeros((1, 2, 16, 18), dtype=torch.float32, device="cuda")[..., :16]
    with pytest.raises(agb.AttnError):
        agb.attn_fwd(q, q, q, bias=bias)
