"""fp64 CPU oracle for the fused attention forward pass -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
binding) never loads it and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64).  This module only
compiles it with gcc, loads it with ctypes and marshals numpy arrays.

What each function restates:
  * :func:`attention`, :func:`attention_rows`, :func:`probs` -- exact attention,
    "Fused attention kernel" (wikillm concept card), Overview and
    Implementation sketch: O = softmax(scale * Q K^T) V per sequence (causal:
    top-left aligned), lse = M + log Z in natural-log units;
  * :func:`attention_rows_gqa`, :func:`attention_gqa`,
    :func:`attention_varlen_gqa`, :func:`attention_paged` -- the same
    definition for the inference variants (HippoAttention case study,
    streamhpc.com, "Our approach": paged attention; FlashAttention-3 summary,
    arxivlens, Limitations: LLM inference): grouped K/V heads, query and key
    sequences of different lengths (causal: queries at the end), keys read
    through a page table;
  * :func:`merge_partials` -- the combination of softmax results over
    disjoint key sets (split-key decoding), written out from the definition;
  * :func:`attention_backward` -- the gradients of that definition with
    respect to Q, K and V, written out from the chain rule (the backward pass
    the FlashAttention-3 summary's Key Results and the card's "When to use
    which" refer to); :func:`attention_backward_rows` gives selected rows of
    the same gradients for one sequence and K/V head at any length;
  * :func:`attention_bias` -- the same definition with an additive bias on
    the scores (the "[+mask]" of the problem statement; "Bias" among the
    additions of the HippoAttention case study, "Our approach");
  * :func:`rotate`, :func:`hadamard_matrix` -- incoherent processing, same card,
    "8-bit forward pass (FP8, Hopper)": x -> x * diag(signs) * H_d / sqrt(d);
  * :func:`e4m3_encode`, :func:`e4m3_decode`, :func:`block_quant`,
    :func:`quantize_qkv` -- e4m3 block quantisation, same section: one scale
    per 128-token block of one (batch, head), scale = amax / 448.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

_lib = None
_lock = threading.Lock()

_dp = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i8p = ctypes.POINTER(ctypes.c_int8)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/_build/liboracle.so (portable C, no
    architecture-specific flags)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                           "-lm", "-lpthread"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_attention_rows.argtypes = [
            _dp, _dp, _dp, _i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_double, ctypes.c_int32, _i64p, _i32p, ctypes.c_int64, _dp, _dp,
            ctypes.c_int32]
        lib.oracle_attention_rows_gqa.argtypes = [
            _dp, _dp, _dp, _i32p, _i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, ctypes.c_double, ctypes.c_int32, _i64p, _i32p, ctypes.c_int64, _dp,
            _dp, ctypes.c_int32]
        lib.oracle_attention_rows_bias.argtypes = [
            _dp, _dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _i32p, _i32p,
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
            ctypes.c_int32, _i64p, _i32p, ctypes.c_int64, _dp, _dp, ctypes.c_int32]
        lib.oracle_attention_backward.argtypes = [
            _dp, _dp, _dp, _dp, _i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, ctypes.c_double, ctypes.c_int32, _dp, _dp, _dp, ctypes.c_int32]
        lib.oracle_attention_backward_rows.argtypes = [
            _dp, _dp, _dp, _dp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_double, ctypes.c_int32, ctypes.c_int32, _i64p, ctypes.c_int32, _i64p,
            ctypes.c_int32, _dp, _dp, _dp, ctypes.c_int32]
        lib.oracle_merge_partials.argtypes = [_dp, _dp, ctypes.c_int32, ctypes.c_int64,
                                              ctypes.c_int32, _dp, _dp]
        lib.oracle_attention_probs.argtypes = [
            _dp, _dp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
            ctypes.c_int32, _dp]
        lib.oracle_hadamard_matrix.argtypes = [ctypes.c_int32, _dp]
        lib.oracle_rotate.argtypes = [_dp, ctypes.c_int64, ctypes.c_int32, _i8p, _dp]
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode_array.argtypes = [_dp, ctypes.c_int64, _u8p]
        lib.oracle_e4m3_decode_array.argtypes = [_u8p, ctypes.c_int64, _dp]
        lib.oracle_block_quant.argtypes = [
            _dp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, ctypes.c_int32, _u8p, _dp]
        _lib = lib
        return lib


def _f64(x) -> np.ndarray:
    """Exact up-conversion to a contiguous float64 array (accepts numpy arrays
    and CPU torch tensors of any float dtype, bf16/fp16 included)."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def attention_rows(q, k, v, cu_seqlens, scale: float, causal: bool, row_tok, row_head,
                   nthreads: int | None = None):
    """O [nrows, d] and lse [nrows] for the packed layout q, k, v [T, H, d]."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, d = q.shape
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    rt = np.ascontiguousarray(row_tok, dtype=np.int64)
    rh = np.ascontiguousarray(row_head, dtype=np.int32)
    n = rt.shape[0]
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    rc = lib.oracle_attention_rows(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(cu, _i32p),
                                   len(cu) - 1, H, d, float(scale), int(bool(causal)),
                                   _ptr(rt, _i64p), _ptr(rh, _i32p), n,
                                   _ptr(o, _dp), _ptr(lse, _dp),
                                   nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attention_rows failed ({rc})")
    return o, lse


def attention_varlen(q, k, v, cu_seqlens, scale: float, causal: bool, nthreads=None):
    """Full O [T, H, d] and lse [H, T] for packed sequences."""
    q = _f64(q)
    T, H, d = q.shape
    tok = np.repeat(np.arange(T, dtype=np.int64), H)
    head = np.tile(np.arange(H, dtype=np.int32), T)
    o, lse = attention_rows(q, k, v, cu_seqlens, scale, causal, tok, head, nthreads)
    return o.reshape(T, H, d), lse.reshape(T, H).T.copy()


def attention(q, k, v, scale: float, causal: bool, nthreads=None):
    """Full O [B, N, H, d] and lse [B, H, N] for a dense batch [B, N, H, d]."""
    q = _f64(q)
    B, N, H, d = q.shape
    cu = (np.arange(B + 1) * N).astype(np.int32)
    o, lse = attention_varlen(q.reshape(B * N, H, d), _f64(k).reshape(B * N, H, d),
                              _f64(v).reshape(B * N, H, d), cu, scale, causal, nthreads)
    return o.reshape(B, N, H, d), lse.reshape(H, B, N).transpose(1, 0, 2).copy()


def attention_rows_gqa(q, k, v, cu_q, cu_k, scale: float, causal: bool, row_tok, row_head,
                       nthreads: int | None = None):
    """O [nrows, d] and lse [nrows] with separate query / key sequences and
    grouped K/V heads: q [Tq, H, d], k, v [Tk, Hkv, d]; sequence s holds
    queries cu_q[s]..cu_q[s+1]-1 and keys cu_k[s]..cu_k[s+1]-1; query head h
    uses K/V head h // (H // Hkv); causal: the queries are the last Lq of the
    Lk positions (query i sees keys j <= i + Lk - Lq)."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, H, d = q.shape
    Hkv = k.shape[1]
    cq = np.ascontiguousarray(cu_q, dtype=np.int32)
    ck = np.ascontiguousarray(cu_k, dtype=np.int32)
    rt = np.ascontiguousarray(row_tok, dtype=np.int64)
    rh = np.ascontiguousarray(row_head, dtype=np.int32)
    n = rt.shape[0]
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    rc = lib.oracle_attention_rows_gqa(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp),
                                       _ptr(cq, _i32p), _ptr(ck, _i32p), len(cq) - 1, H, Hkv, d,
                                       float(scale), int(bool(causal)), _ptr(rt, _i64p),
                                       _ptr(rh, _i32p), n, _ptr(o, _dp), _ptr(lse, _dp),
                                       nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attention_rows_gqa failed ({rc})")
    return o, lse


def attention_varlen_gqa(q, k, v, cu_q, cu_k, scale: float, causal: bool, nthreads=None):
    """Full O [Tq, H, d] and lse [H, Tq] for packed query / key sequences
    with grouped K/V heads (see attention_rows_gqa)."""
    q = _f64(q)
    Tq, H, d = q.shape
    tok = np.repeat(np.arange(Tq, dtype=np.int64), H)
    head = np.tile(np.arange(H, dtype=np.int32), Tq)
    o, lse = attention_rows_gqa(q, k, v, cu_q, cu_k, scale, causal, tok, head, nthreads)
    return o.reshape(Tq, H, d), lse.reshape(Tq, H).T.copy()


def attention_gqa(q, k, v, scale: float, causal: bool, nthreads=None):
    """Dense O [B, Nq, H, d] and lse [B, H, Nq] for q [B, Nq, H, d] and
    k, v [B, Nk, Hkv, d] (causal: the queries are the last Nq positions)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Nq, H, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    cq = (np.arange(B + 1) * Nq).astype(np.int32)
    ck = (np.arange(B + 1) * Nk).astype(np.int32)
    o, lse = attention_varlen_gqa(q.reshape(B * Nq, H, d), k.reshape(B * Nk, Hkv, d),
                                  v.reshape(B * Nk, Hkv, d), cq, ck, scale, causal, nthreads)
    return o.reshape(B, Nq, H, d), lse.reshape(H, B, Nq).transpose(1, 0, 2).copy()


def attention_bias(q, k, v, bias, scale: float, causal: bool, nthreads=None):
    """Dense O [B, N, H, d] and lse [B, H, N] with an additive score bias:
    s_ij = scale * q_i . k_j + bias[b, h, i, j], bias broadcastable to
    [B, H, N, N] (numpy broadcasting over the first two axes; a size-1 row
    axis broadcasts over queries).  -inf removes a key."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    bias = np.asarray(_f64(bias))
    while bias.ndim < 4:
        bias = bias[None]
    sb = 0 if bias.shape[0] == 1 else bias.strides[0] // 8
    sh = 0 if bias.shape[1] == 1 else bias.strides[1] // 8
    sr = 0 if bias.shape[2] == 1 else bias.strides[2] // 8
    if bias.shape[3] != N or bias.strides[3] != 8:
        raise ValueError("bias keys must be the last, contiguous axis of length N")
    cu = (np.arange(B + 1) * N).astype(np.int32)
    tok = np.repeat(np.arange(B * N, dtype=np.int64), H)
    head = np.tile(np.arange(H, dtype=np.int32), B * N)
    o = np.empty((tok.shape[0], d), dtype=np.float64)
    lse = np.empty(tok.shape[0], dtype=np.float64)
    qq, kk, vv = q.reshape(B * N, H, d), k.reshape(B * N, Hkv, d), v.reshape(B * N, Hkv, d)
    rc = lib.oracle_attention_rows_bias(_ptr(qq, _dp), _ptr(kk, _dp), _ptr(vv, _dp),
                                        bias.ctypes.data_as(_dp), sb, sh, sr, _ptr(cu, _i32p),
                                        _ptr(cu, _i32p), B, H, Hkv, d, float(scale),
                                        int(bool(causal)), _ptr(tok, _i64p), _ptr(head, _i32p),
                                        tok.shape[0], _ptr(o, _dp), _ptr(lse, _dp),
                                        nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attention_rows_bias failed ({rc})")
    return o.reshape(B, N, H, d), lse.reshape(B, N, H).transpose(0, 2, 1).copy()


def attention_backward(q, k, v, dout, scale: float, causal: bool, nthreads=None):
    """Gradients (dq, dk, dv) of the dense forward O = softmax(scale Q K^T) V
    for an upstream gradient dout: q, dout [B, N, H, d]; k, v [B, N, Hkv, d]."""
    lib = _load()
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    cu = (np.arange(B + 1) * N).astype(np.int32)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    rc = lib.oracle_attention_backward(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(do, _dp),
                                       _ptr(cu, _i32p), B, H, Hkv, d, float(scale),
                                       int(bool(causal)), _ptr(dq, _dp), _ptr(dk, _dp),
                                       _ptr(dv, _dp), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attention_backward failed ({rc})")
    return dq, dk, dv


def attention_backward_rows(q, k, v, dout, scale: float, causal: bool, hk: int, qrows, krows,
                            nthreads=None):
    """Selected gradient rows of one sequence at any length: q, dout [L, H, d];
    k, v [L, Hkv, d].  Returns dq_rows [g, len(qrows), d] for the g query heads
    of K/V head hk, and dk_rows, dv_rows [len(krows), d] summed over them."""
    lib = _load()
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    L, H, d = q.shape
    Hkv = k.shape[1]
    g = H // Hkv
    qr = np.ascontiguousarray(qrows, dtype=np.int64)
    kr = np.ascontiguousarray(krows, dtype=np.int64)
    dq = np.empty((g, len(qr), d))
    dk = np.empty((len(kr), d))
    dv = np.empty((len(kr), d))
    rc = lib.oracle_attention_backward_rows(
        _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(do, _dp), L, H, Hkv, d, float(scale),
        int(bool(causal)), int(hk), _ptr(qr, _i64p), len(qr), _ptr(kr, _i64p), len(kr),
        _ptr(dq, _dp), _ptr(dk, _dp), _ptr(dv, _dp), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attention_backward_rows failed ({rc})")
    return dq, dk, dv


def gather_pages(cache, block_table, seqlens):
    """The keys (or values) of each sequence of a paged cache, packed:
    cache [num_pages, page_size, Hkv, d]; token t of sequence b is row
    t % page_size of page block_table[b][t // page_size].  Returns
    ([sum(seqlens), Hkv, d], cu) with cu the key offsets."""
    cache = np.asarray(cache)
    P = cache.shape[1]
    rows = []
    for b, L in enumerate(seqlens):
        t = np.arange(int(L))
        rows.append(cache[np.asarray(block_table[b])[t // P], t % P])
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    return np.concatenate(rows, axis=0), cu


def attention_paged(q, k_cache, v_cache, block_table, seqlens_k, scale: float, causal: bool,
                    nthreads=None):
    """O [B, Nq, H, d] and lse [B, H, Nq] of queries q [B, Nq, H, d] against a
    paged K/V cache (see gather_pages); causal: the Nq queries are the last
    Nq of the seqlens_k[b] positions."""
    q = _f64(q)
    B, Nq, H, d = q.shape
    kp, ck = gather_pages(_f64(k_cache), block_table, seqlens_k)
    vp, _ = gather_pages(_f64(v_cache), block_table, seqlens_k)
    cq = (np.arange(B + 1) * Nq).astype(np.int32)
    o, lse = attention_varlen_gqa(q.reshape(B * Nq, H, d), kp, vp, cq, ck, scale, causal,
                                  nthreads)
    return o.reshape(B, Nq, H, d), lse.reshape(H, B, Nq).transpose(1, 0, 2).copy()


def merge_partials(o_parts, lse_parts):
    """Combine results over disjoint key sets of the same rows:
    o_parts [S, R, d], lse_parts [S, R] -> (o [R, d], lse [R]) with
    lse = log sum_s exp(lse_s) and O = sum_s exp(lse_s - lse) O_s."""
    lib = _load()
    op = _f64(o_parts)
    lp = _f64(lse_parts)
    S, R, d = op.shape
    o = np.empty((R, d), dtype=np.float64)
    lse = np.empty(R, dtype=np.float64)
    if lib.oracle_merge_partials(_ptr(op, _dp), _ptr(lp, _dp), S, R, d, _ptr(o, _dp),
                                 _ptr(lse, _dp)) != 0:
        raise ValueError("oracle_merge_partials failed")
    return o, lse


def probs(q, k, scale: float, causal: bool):
    """P [H, N, N] of one sequence q, k [N, H, d] (small shapes only)."""
    lib = _load()
    q, k = _f64(q), _f64(k)
    N, H, d = q.shape
    p = np.empty((H, N, N), dtype=np.float64)
    rc = lib.oracle_attention_probs(_ptr(q, _dp), _ptr(k, _dp), N, H, d, float(scale),
                                    int(bool(causal)), _ptr(p, _dp))
    if rc != 0:
        raise ValueError("oracle_attention_probs failed")
    return p


def hadamard_matrix(d: int) -> np.ndarray:
    lib = _load()
    hm = np.empty((d, d), dtype=np.float64)
    if lib.oracle_hadamard_matrix(d, _ptr(hm, _dp)) != 0:
        raise ValueError("d must be a power of two")
    return hm


def rotate(x, signs) -> np.ndarray:
    """x [..., d] -> x * diag(signs) * H_d / sqrt(d) (signs None: no sign flip)."""
    lib = _load()
    x = _f64(x)
    d = x.shape[-1]
    flat = x.reshape(-1, d)
    out = np.empty_like(flat)
    sg = None if signs is None else np.ascontiguousarray(signs, dtype=np.int8)
    rc = lib.oracle_rotate(_ptr(flat, _dp), flat.shape[0], d,
                           None if sg is None else _ptr(sg, _i8p), _ptr(out, _dp))
    if rc != 0:
        raise ValueError("oracle_rotate failed")
    return out.reshape(x.shape)


def e4m3_encode(x) -> np.ndarray:
    lib = _load()
    x = _f64(x)
    flat = x.reshape(-1)
    out = np.empty(flat.shape[0], dtype=np.uint8)
    lib.oracle_e4m3_encode_array(_ptr(flat, _dp), flat.shape[0], _ptr(out, _u8p))
    return out.reshape(x.shape)


def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    flat = c.reshape(-1)
    out = np.empty(flat.shape[0], dtype=np.float64)
    lib.oracle_e4m3_decode_array(_ptr(flat, _u8p), flat.shape[0], _ptr(out, _dp))
    return out.reshape(c.shape)


def block_quant(x, per_tensor: bool = False, block: int = 128):
    """codes uint8 [B,N,H,d] and descale float64 [B,H,ceil(N/block)] of x [B,N,H,d]."""
    lib = _load()
    x = _f64(x)
    B, N, H, d = x.shape
    nblk = (N + block - 1) // block
    codes = np.empty(x.shape, dtype=np.uint8)
    desc = np.empty((B, H, nblk), dtype=np.float64)
    rc = lib.oracle_block_quant(_ptr(x, _dp), B, N, H, d, block, int(bool(per_tensor)),
                                _ptr(codes, _u8p), _ptr(desc, _dp))
    if rc != 0:
        raise ValueError("oracle_block_quant failed")
    return codes, desc


def quantize_qkv(q, k, v, signs, per_tensor: bool = False, block: int = 128):
    """The fp8 pre-step in the pages' order: rotate Q and K by
    diag(signs) * H_d / sqrt(d) (skipped when signs is None), then quantise Q,
    K and V to e4m3 with block (or per-tensor) scales.  Returns a dict with the
    codes, descales and the rotated fp64 values that were quantised."""
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    if signs is not None:
        qf, kf = rotate(qf, signs), rotate(kf, signs)
    out = {"q_rot": qf, "k_rot": kf}
    for nm, x in (("q", qf), ("k", kf), ("v", vf)):
        out[nm + "8"], out["d" + nm] = block_quant(x, per_tensor, block)
    return out


def dequantize(codes, descale, block: int = 128) -> np.ndarray:
    """decode(code) * descale of its block, [B,N,H,d]."""
    x = e4m3_decode(codes)
    B, N, H, d = x.shape
    blk = np.arange(N) // block
    s = np.asarray(descale, dtype=np.float64)[:, :, blk]          # [B, H, N]
    return x * s.transpose(0, 2, 1)[..., None]
