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
    hst = L.attn_fwd_host
    assert hst(None, FAKE, FAKE, FAKE, None, 2, 4, 16, 64, 0.1, 0, 0, None) == 1
    assert hst(FAKE, FAKE, FAKE, FAKE, None, 0, 4, 16, 64, 0.1, 0, 0, None) == 1
    assert hst(FAKE, FAKE, FAKE, FAKE, None, 2, 4, 16, 96, 0.1, 0, 0, None) == 2
    assert hst(FAKE, FAKE, FAKE + 4, FAKE, None, 2, 4, 16, 64, 0.1, 0, 0, None) == 3
    fh = L.attn_fwd_fp8_host
    #        q     k     v     signs o     lse   B  H  N   d    scale causal stream
    assert fh(None, FAKE, FAKE, None, FAKE, None, 2, 4, 16, 128, 0.1, 0, None) == 1
    assert fh(FAKE, FAKE, FAKE, None, FAKE, None, 2, 4, 0, 128, 0.1, 0, None) == 1
    assert fh(FAKE, FAKE, FAKE, None, FAKE, None, 2, 4, 16, 96, 0.1, 0, None) == 2
    assert fh(FAKE, FAKE, FAKE, None, FAKE + 4, None, 2, 4, 16, 128, 0.1, 0, None) == 3
    f = L.attn_fwd_fp8
    assert f(FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, 1, 1, 16, 128, 0.1, 0, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 1, 16, 96, 0.1, 0, None) == 2
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


def test_gqa_entry_points_reject_bad_head_counts(L):
    g = L.attn_fwd_gqa
    #       q     k     v     o     lse   B  H  Hkv N   d   scale causal dtype stream
    assert g(FAKE, FAKE, FAKE, FAKE, None, 1, 8, 0, 16, 64, 0.125, 0, 0, None) == 1
    assert g(FAKE, FAKE, FAKE, FAKE, None, 1, 8, 3, 16, 64, 0.125, 0, 0, None) == 1
    assert g(FAKE, FAKE, FAKE, FAKE, None, 1, 8, 16, 16, 64, 0.125, 0, 0, None) == 1
    assert g(FAKE, FAKE, FAKE, FAKE, None, 1, 8, 2, 16, 96, 0.125, 0, 0, None) == 2
    gv = L.attn_fwd_varlen_gqa
    assert gv(FAKE, FAKE, FAKE, FAKE, None, FAKE, 2, 10, 8, 8, 3, 64, 0.1, 1, 0, None) == 1
    assert gv(FAKE, FAKE, FAKE, FAKE, None, None, 2, 10, 8, 8, 2, 64, 0.1, 1, 0, None) == 1


def test_paged_entry_point_rejects_bad_arguments(L):
    p = L.attn_fwd_paged
    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, o=FAKE, lse=None, B=1, Nq=1, H=8,
                 Hkv=2, d=128, P=16, maxp=4, npages=8, maxk=64, scale=0.1, causal=1, dtype=0,
                 splits=0, stream=None)
        a.update(kw)
        return p(a["q"], a["k"], a["v"], a["bt"], a["sl"], a["o"], a["lse"], a["B"], a["Nq"],
                 a["H"], a["Hkv"], a["d"], a["P"], a["maxp"], a["npages"], a["maxk"],
                 a["scale"], a["causal"], a["dtype"], a["splits"], a["stream"])
    assert call(bt=None) == 1
    assert call(Hkv=3) == 1
    assert call(maxk=65) == 1            # more keys than the table can name
    assert call(splits=-1) == 1
    assert call(d=96) == 2
    assert call(Nq=4, H=8, Hkv=1) == 2   # 32 query rows per K/V head
    assert call(q=FAKE + 4) == 3
