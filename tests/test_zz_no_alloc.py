"""attn_fwd_varlen_noalloc: the varlen forward pass for callers that cannot
allocate device memory (plugins whose device memory a host framework plans,
services that forbid allocation after start-up).  Called through the C ABI
with caller-owned buffers; its output must agree with the regular
attn_fwd_varlen within the parity tolerances (O 2e-3, lse 1e-3), on two calls
in a row that reuse the shared static scratch.

Kept in a file pytest collects last, so a stop-at-first-failure run has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import attention_forward_softmax_gb300 as agb
from tests._gpu_helpers import TOL_LSE, TOL_O, qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    agb.build()
    return agb.lib()


def call_noalloc(L, q, k, v, o, lse, cu, max_seqlen, causal, status):
    T, H, d = q.shape
    stream = torch.cuda.current_stream().cuda_stream
    return L.attn_fwd_varlen_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), cu.data_ptr(), cu.numel() - 1, T,
                                     int(max_seqlen), H, d, ctypes.c_float(d ** -0.5),
                                     int(causal), 0, status.data_ptr(), stream)


def problem(lens, H, d, seed):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v = (t.cuda() for t in qkv(seed, (T, H, d), torch.bfloat16))
    return q, k, v, torch.from_numpy(cu).cuda(), max(lens)


def test_noalloc_matches_regular_entry_point_on_two_calls(L):
    cases = [([300, 17, 1024, 129, 5], 4, 128, True, 3100),
             ([64, 700, 256, 2000], 2, 64, False, 3101)]
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for lens, H, d, causal, seed in cases:
        q, k, v, cu, mx = problem(lens, H, d, seed)
        T = q.shape[0]
        o_ref, lse_ref = agb.attn_fwd_varlen(q, k, v, cu, mx, causal=causal)
        o = torch.empty_like(q)
        lse = torch.empty((H, T), dtype=torch.float32, device="cuda")
        rc = call_noalloc(L, q, k, v, o, lse, cu, mx, causal, status)
        assert rc == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert float((o.float() - o_ref.float()).abs().max()) <= TOL_O
        assert float((lse - lse_ref).abs().max()) <= TOL_LSE


def test_noalloc_status_and_size_limit(L):
    q, k, v, cu, mx = problem([40, 40], 1, 64, 3102)
    o = torch.empty_like(q)
    lse = torch.empty((1, q.shape[0]), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = torch.tensor([0, 50, 30], dtype=torch.int32, device="cuda")      # decreasing
    assert call_noalloc(L, q, k, v, o, lse, bad, 60, True, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 6                                     # ATTN_ERR_BAD_SEQLENS
    assert call_noalloc(L, q, k, v, o, lse, cu, mx, True, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0                                     # reset by the call
    # beyond the fixed tile-list capacity: rejected on the host, nothing launched
    big_T = 256 * 40000
    rc = L.attn_fwd_varlen_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None,
                                   cu.data_ptr(), 1, big_T, big_T, 1, 64, ctypes.c_float(0.125),
                                   0, 0, None, None)
    assert rc == 8                                                     # ATTN_ERR_TOO_LARGE
