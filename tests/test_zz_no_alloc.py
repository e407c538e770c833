"""attn_fwd_varlen_noalloc: the varlen forward pass for callers that cannot
allocate device memory (plugins whose device memory a host framework plans,
services that forbid allocation after start-up).  Called through the C ABI
with caller-owned buffers.

It runs the same kernels on the same tile list as the regular
attn_fwd_varlen, and each work tile is computed the same way whichever CTA
takes it, so its output must be bitwise equal to the regular entry point's,
on two calls in a row that reuse the shared static scratch.  A second case
runs in a fresh process that never calls the allocating entry points: the
output matches the fp64 oracle within the parity tolerances, and repeated
calls leave the device's free memory unchanged.

Kept in a file pytest collects last, so a stop-at-first-failure run has
already run every other test."""
import ast
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import attention_forward_softmax_gb300 as agb
from tests._gpu_helpers import qkv

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


def test_noalloc_matches_regular_entry_point_bitwise_on_two_calls(L):
    cases = [([300, 17, 1024, 129, 5], 4, 128, True, 3100),
             ([64, 700, 256, 2000], 2, 64, False, 3101)]
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for lens, H, d, causal, seed in cases:
        q, k, v, cu, mx = problem(lens, H, d, seed)
        T = q.shape[0]
        o_ref, lse_ref = agb.attn_fwd_varlen(q, k, v, cu, mx, causal=causal)
        o = torch.full_like(q, float("nan"))
        lse = torch.full((H, T), float("nan"), dtype=torch.float32, device="cuda")
        assert call_noalloc(L, q, k, v, o, lse, cu, mx, causal, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))


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


# A fresh process in which only the no-alloc entry point is ever called.  Its
# inputs, outputs and status word are allocated up front; then three calls:
# the first one loads the kernels, the next two must not change the device's
# free memory.
CHILD = r"""
import ctypes, math, sys
import numpy as np, torch
import attention_forward_softmax_gb300 as agb
from tests._gpu_helpers import TOL_LSE, o_tolerance, oracle_varlen, qkv
L = agb.lib()
lens = [200, 1, 333, 64]
H, d = 3, 128
cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
T = int(cu[-1])
q, k, v = qkv(3103, (T, H, d), torch.bfloat16)
qd, kd, vd = (t.cuda() for t in (q, k, v))
cud = torch.from_numpy(cu).cuda()
o = torch.empty_like(qd)
lse = torch.empty((H, T), dtype=torch.float32, device="cuda")
status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
stream = torch.cuda.current_stream().cuda_stream
def call():
    rc = L.attn_fwd_varlen_noalloc(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), cud.data_ptr(), len(lens), T, max(lens), H, d,
                                   ctypes.c_float(d ** -0.5), 1, 0, status.data_ptr(), stream)
    torch.cuda.synchronize()
    assert rc == 0 and int(status.item()) == 0, (rc, int(status.item()))
call()
free = []
for _ in range(2):
    free.append(torch.cuda.mem_get_info()[0])
    call()
free.append(torch.cuda.mem_get_info()[0])
o_ref, lse_ref, a_ref, ne = oracle_varlen(q, k, v, cu, 1 / math.sqrt(d), True)
tol = o_tolerance(o_ref, a_ref, torch.bfloat16, ne)
err = np.abs(o.float().cpu().numpy() - o_ref)
assert np.all(err <= tol), float(err.max())
assert float(np.abs(lse.cpu().numpy() - lse_ref).max()) <= TOL_LSE
print("FREE", free)
print("CHILD OK")
"""


def test_noalloc_alone_in_a_fresh_process():
    agb.build()
    r = subprocess.run([sys.executable, "-c", CHILD], env=dict(os.environ, PYTHONPATH=ROOT),
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "CHILD OK" in r.stdout
    free = ast.literal_eval(r.stdout.split("FREE", 1)[1].splitlines()[0].strip())
    assert len(set(free)) == 1, free
