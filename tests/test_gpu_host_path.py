"""attn_fwd_host: the dense forward on host buffers, copies of one chunk
(a batch entry, or a group of heads of the first and last entries)
overlapped with the compute of earlier chunks.  It runs the same kernel on
each chunk that attn_fwd runs on the whole batch, without splitting the last
wave; at shapes where attn_fwd splits nothing either, every tile is
computed the same way: the outputs must be bitwise equal to attn_fwd's on
device copies of the same inputs.  Also: head-group chunks, pageable host
memory, no lse, B = 1, and stream order (work queued after the call sees
the outputs)."""
import numpy as np
import pytest
import torch

import attention_forward_softmax_gb300 as agb
from datagen import random_signs
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


def no_split(B, H, N):
    """attn_fwd leaves every tile whole at this shape (non-causal)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = B * H * ((N + 255) // 256)
    grid = min(T, sms)
    rem = T % grid
    return rem == 0 or 2 * rem > grid


@pytest.mark.parametrize("B,H,N,causal", [(2, 32, 4096, False), (3, 48, 4096, True),
                                             (1, 32, 4096, True)])
def test_host_path_head_group_chunks(B, H, N, causal):
    """Shapes whose 256-row tiles fill the SMs with fewer heads than H, so
    the first and last entries move as head groups (strided 2-D copies)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nqt = (N + 255) // 256
    assert any(H % x == 0 and x * nqt >= sms for x in range(1, H)), "no head groups here"
    if not causal and not no_split(B, H, N):
        pytest.skip("attn_fwd would split the last wave at this SM count")
    q, k, v = qkv(9530 + H, (B, N, H, 128), torch.bfloat16)
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


def fp8_device_reference(q, k, v, signs, causal):
    q8, k8, v8, dq, dk, dv = agb.qkv_block_quant_hadamard(
        q.cuda(), k.cuda(), v.cuda(), None if signs is None else signs.cuda())
    o, lse = agb.attn_fwd_fp8(q8, k8, v8, dq, dk, dv, causal=causal)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def fp8_no_split(B, H, N, d):
    """attn_fwd_fp8 leaves every tile whole at this shape (non-causal)."""
    return d != 128 or no_split(B, H, N)


@pytest.mark.parametrize("B,H,N,d,causal,rot", [
    (2, 32, 4096, 128, False, True),      # head groups at both ends
    (3, 48, 4096, 128, True, True),
    (3, 4, 700, 128, False, False),       # whole entries, ragged blocks, no rotation
    (2, 3, 300, 64, True, True),
    (1, 32, 4096, 128, True, True),       # one entry, cut into head groups
])
def test_fp8_host_path_matches_device_path_bitwise(B, H, N, d, causal, rot):
    """attn_fwd_fp8_host quantises each chunk (block scales per (b, h,
    128-token block): the same codes and scales as the whole tensor) and runs
    the e4m3 kernel on it; at shapes where attn_fwd_fp8 splits nothing the
    outputs are bitwise those of the device path."""
    if not causal and not fp8_no_split(B, H, N, d):
        pytest.skip("attn_fwd_fp8 would split the last wave at this SM count")
    q, k, v = qkv(9540 + H + d, (B, N, H, d), torch.bfloat16)
    signs = torch.from_numpy(random_signs(9541, d)) if rot else None
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o, lse = agb.attn_fwd_fp8_host(hq, hk, hv, signs=signs, causal=causal)
    torch.cuda.current_stream().synchronize()
    assert agb.get_status() == 0
    o_ref, lse_ref = fp8_device_reference(q, k, v, signs, causal)
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))
