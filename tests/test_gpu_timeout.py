"""Failure detection without a GPU fault: with a one-cycle wait budget the
kernel's pipeline waits expire at once; it must record ATTN_ERR_TIMEOUT,
drain its own copies and MMAs, free TMEM and return, leaving the CUDA
context usable.  Runs in a child process (the budget is read once per
process from ATTN_WAIT_BUDGET_CYCLES)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import torch
import attention_forward_softmax_gb300 as agb
q = torch.randn(2, 2048, 8, 128, device="cuda").to(torch.bfloat16)
agb.attn_fwd(q, q, q, causal=True)
print("STATUS", agb.get_status())
print("AGAIN", agb.get_status())
x = torch.ones(16, device="cuda")
print("CTX", float(x.sum()))
"""


# the 8-bit path: the quantise kernel (double-buffered copies) and the e4m3
# attention kernel (two softmax warps per row that leave together through
# their pair barrier)
CHILD_FP8 = r"""
import torch
import attention_forward_softmax_gb300 as agb
x = torch.randn(2, 2048, 8, 128, device="cuda").to(torch.bfloat16)
q8, k8, v8, dq, dk, dv = agb.qkv_block_quant_hadamard(x, x, x, None)
agb.attn_fwd_fp8(q8, k8, v8, dq, dk, dv, causal=False)
print("STATUS", agb.get_status())
print("AGAIN", agb.get_status())
y = torch.ones(16, device="cuda")
print("CTX", float(y.sum()))
"""


# the backward kernel: five roles (copies, MMAs, two groups of warps that
# leave their loops together through named barriers, dQ bulk reduces)
CHILD_BWD = r"""
import torch
import attention_forward_softmax_gb300 as agb
x = torch.randn(1, 1024, 4, 128, device="cuda").to(torch.bfloat16)
lse = torch.zeros(1, 4, 1024, device="cuda")
agb.attn_bwd(x, x, x, x, lse, x, causal=True)
print("STATUS", agb.get_status())
print("AGAIN", agb.get_status())
y = torch.ones(16, device="cuda")
print("CTX", float(y.sum()))
"""


# paged decoding with 64-row pages: the tensor-copy path.  Its only waits
# are for copies, and a wait's first probe suspends until the copy lands, so
# even a one-cycle budget need not expire; the call must still complete,
# report either no error or ATTN_ERR_TIMEOUT, and leave the context usable.
CHILD_PAGED = r"""
import torch
import attention_forward_softmax_gb300 as agb
kc = torch.randn(512, 64, 8, 128, device="cuda").to(torch.bfloat16)
q = torch.randn(8, 1, 32, 128, device="cuda").to(torch.bfloat16)
table = torch.randperm(512, device="cuda").to(torch.int32).reshape(8, 64).contiguous()
seql = torch.full((8,), 4096, dtype=torch.int32, device="cuda")
agb.attn_fwd_paged(q, kc, kc, table, seql, 4096)
print("STATUS", agb.get_status())
print("AGAIN", agb.get_status())
y = torch.ones(16, device="cuda")
print("CTX", float(y.sum()))
"""


@pytest.mark.parametrize("child", [CHILD, CHILD_FP8, CHILD_BWD, CHILD_PAGED],
                         ids=["bf16", "fp8", "bwd", "paged"])
def test_wait_timeout_is_reported_and_context_survives(child):
    env = dict(os.environ, ATTN_WAIT_BUDGET_CYCLES="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", child], env=env, capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    if child is CHILD_PAGED:
        assert "STATUS 5" in r.stdout or "STATUS 0" in r.stdout, r.stdout
    else:
        assert "STATUS 5" in r.stdout, r.stdout
    assert "AGAIN 0" in r.stdout, r.stdout
    assert "CTX 16.0" in r.stdout, r.stdout
