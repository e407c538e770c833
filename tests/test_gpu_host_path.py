"""attn_fwd_host: the dense forward on host buffers, copies of one batch
entry overlapped with the compute of the previous one.  It runs the same
kernel on each batch entry that attn_fwd runs on the whole batch, and at
these sizes (fewer work tiles than SMs, so no tile is split) every tile is
computed the same way: the outputs must be bitwise equal to attn_fwd's on
device copies of the same inputs.  Also: pageable host memory, no lse,
B = 1, and stream order (work queued after the call sees the outputs)."""
import numpy as np
import pytest
import torch

import attention_forward_softmax_gb300 as agb
from tests._gpu_helpers import qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    agb.build()
    agb.lib()


def device_reference(q, k, v, causal):
    o, lse = agb.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("B,N,H,d,dtype,causal", [
    (3, 700, 4, 128, torch.bfloat16, True),
    (4, 513, 2, 64, torch.float16, False),
    (1, 300, 3, 128, torch.bfloat16, False),
])
def test_host_path_matches_device_path_bitwise(B, N, H, d, dtype, causal):
    q, k, v = qkv(9500 + N, (B, N, H, d), dtype)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o, lse = agb.attn_fwd_host(hq, hk, hv, causal=causal)
    torch.cuda.current_stream().synchronize()
    assert agb.get_status() == 0
    o_ref, lse_ref = device_reference(q, k, v, causal)
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))


def test_host_path_pageable_memory_and_no_lse():
    B, N, H, d = 3, 400, 2, 64
    q, k, v = qkv(9510, (B, N, H, d), torch.bfloat16)      # pageable
    o, lse = agb.attn_fwd_host(q, k, v, causal=True, want_lse=False)
    torch.cuda.current_stream().synchronize()
    assert lse is None and agb.get_status() == 0
    o_ref, _ = device_reference(q, k, v, True)
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))


def test_host_path_outputs_are_ordered_on_the_stream():
    """A device copy of the output queued on the same stream right after the
    call sees the finished values."""
    B, N, H, d = 4, 600, 2, 128
    q, k, v = qkv(9520, (B, N, H, d), torch.bfloat16)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = agb.attn_fwd_host(hq, hk, hv, causal=False, stream=s)
        o_dev = o.to("cuda", non_blocking=True)        # queued on s after the call
    s.synchronize()
    o_ref, _ = device_reference(q, k, v, False)
    assert torch.equal(o_dev.cpu().view(torch.int16), o_ref.view(torch.int16))
    assert np.isfinite(lse.numpy()).all()
