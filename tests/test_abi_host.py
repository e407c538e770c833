"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/attn.h declares, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

import attention_forward_softmax_gb300 as agb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    agb.build()
    return agb.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_expected_calls():
    names = declared_functions()
    for nm in ("attn_fwd", "attn_fwd_varlen", "attn_fwd_fp8", "qkv_block_quant_hadamard",
               "attn_get_status"):
        assert nm in names


def test_library_exports_every_declared_symbol(L):
    for nm in declared_functions():
        assert hasattr(L, nm), nm


def test_version_and_status_strings(L):
    assert L.attn_version() == 0x100
    for code in range(9):
        assert L.attn_status_string(code)
    assert L.attn_status_string(0) == b"ok"
    assert L.attn_status_string(999) == b"unknown status"


FAKE = 1 << 20        # aligned, never dereferenced: validation fails first


def fwd(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, H=1, N=16, d=64, scale=0.125,
             causal=0, dtype=0, stream=None)
    a.update(kw)
    return L.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"],
                      a["scale"], a["causal"], a["dtype"], a["stream"])


def test_attn_fwd_rejects_bad_arguments(L):
    assert fwd(L, q=None) == 1
    assert fwd(L, o=None) == 1
    assert fwd(L, B=0) == 1
    assert fwd(L, H=0) == 1
    assert fwd(L, N=0) == 1
    assert fwd(L, scale=float("nan")) == 1
    assert fwd(L, scale=float("inf")) == 1
    assert fwd(L, d=96) == 2
    assert fwd(L, d=256) == 2
    assert fwd(L, dtype=7) == 2
    assert fwd(L, k=FAKE + 8) == 3
    assert fwd(L, lse=FAKE + 2) == 3


def test_varlen_fp8_quant_reject_bad_arguments(L):
    v = L.attn_fwd_varlen
    assert v(FAKE, FAKE, FAKE, FAKE, None, None, 2, 10, 8, 1, 64, 0.1, 1, 0, None) == 1
    assert v(FAKE, FAKE, FAKE, FAKE, None, FAKE, 0, 10, 8, 1, 64, 0.1, 1, 0, None) == 1
    assert v(FAKE, FAKE, FAKE, FAKE, None, FAKE, 2, 10, 8, 1, 80, 0.1, 1, 0, None) == 2
    assert v(FAKE, FAKE, FAKE, FAKE, None, FAKE + 2, 2, 10, 8, 1, 64, 0.1, 1, 0, None) == 3
    f = L.attn_fwd_fp8
    assert f(FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, 1, 1, 16, 128, 0.1, 0, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 1, 16, 64, 0.1, 0, None) == 2
    qz = L.qkv_block_quant_hadamard
    assert qz(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 0, 1, 1, 16, 64, None) == 1
    assert qz(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, 1, 1, 16, 48, None) == 2
    assert qz(FAKE, FAKE, FAKE, FAKE + 4, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, 1, 1, 16, 64,
              None) == 3


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    """The product path has no fallback: a missing library is an error."""
    monkeypatch.setattr(agb, "_lib", None)
    monkeypatch.setattr(agb, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        agb.lib()
