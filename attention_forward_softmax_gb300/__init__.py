"""GB300 (sm_103a) fused attention forward: Python binding of libattn_gb300.so.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI (``include/attn.h``).  PyTorch supplies device
memory and the current stream.  There is no CPU path: if the library is not
built, every call raises.

    o, lse = attn_fwd(q, k, v, causal=False)                       # [B,N,H,d]
    o, lse = attn_fwd_varlen(q, k, v, cu_seqlens, max_seqlen)      # [T,H,d]
    q8, k8, v8, dq, dk, dv = qkv_block_quant_hadamard(q, k, v, signs)
    o, lse = attn_fwd_fp8(q8, k8, v8, dq, dk, dv)
    o, lse = attn_fwd_paged(q, k_cache, v_cache, block_table, seqlens_k, max_seqlen_k)
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libattn_gb300.so")

ATTN_BF16, ATTN_FP16 = 0, 1
STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
          3: "ATTN_ERR_MISALIGNED", 4: "ATTN_ERR_LAUNCH", 5: "ATTN_ERR_TIMEOUT",
          6: "ATTN_ERR_BAD_SEQLENS", 7: "ATTN_ERR_CUDA", 8: "ATTN_ERR_TOO_LARGE"}
EXPORTS = ("attn_fwd", "attn_fwd_varlen", "attn_fwd_fp8", "qkv_block_quant_hadamard",
           "attn_get_status", "attn_fwd_varlen_noalloc", "attn_fwd_gqa", "attn_fwd_varlen_gqa",
           "attn_fwd_paged", "attn_fwd_bias", "attn_bwd", "attn_fwd_host", "attn_fwd_fp8_host",
           "attn_status_string", "attn_shutdown", "attn_version")

_lib = None
_lock = threading.Lock()


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


def build(force: bool = False) -> str:
    from ._builder import build as _build
    return _build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"CUDA library not built ({LIB_PATH} missing); "
                                   "run attention_forward_softmax_gb300.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
            L.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
            L.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
            L.qkv_block_quant_hadamard.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i,
                                                   i, i, i, i, vp]
            L.attn_fwd_varlen_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i,
                                                  i, vp, vp]
            L.attn_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
            L.attn_fwd_varlen_gqa.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i,
                                              vp]
            L.attn_get_status.argtypes = [vp]
            L.attn_status_string.argtypes = [i]
            L.attn_status_string.restype = ctypes.c_char_p
            L.attn_version.restype = ctypes.c_uint32
            L.attn_fwd_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i,
                                         i, f, i, i, i, vp]
            ll = ctypes.c_longlong
            L.attn_fwd_bias.argtypes = [vp, vp, vp, vp, ll, ll, ll, vp, vp, i, i, i, i, i, f, i, i,
                                        vp]
            L.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
            L.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
            L.attn_fwd_fp8_host.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
            for nm in EXPORTS[:13]:
                getattr(L, nm).restype = ctypes.c_int
            _lib = L
        return _lib


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(rc: int, where: str):
    if rc != 0:
        raise AttnError(rc, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float16:
        return ATTN_FP16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
             want_lse: bool = True, stream=None, bias=None):
    """Dense attention, q [B, N, H, d], k/v [B, N, H_kv, d] (H_kv divides H;
    H_kv < H is grouped-query attention), bf16 or fp16
    -> (o [B,N,H,d], lse [B,H,N] fp32).  `bias`: optional fp32 tensor
    broadcastable to [B, H, N, N] added to the scaled scores."""
    _need_cuda(q, k, v)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if (k.shape != (B, N, Hkv, d) or v.shape != k.shape or k.dtype != q.dtype
            or v.dtype != q.dtype):
        raise ValueError("q [B,N,H,d] and k, v [B,N,H_kv,d] must agree in shape and dtype")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    _need_cuda(o, lse)
    if bias is not None:
        if bias.dtype != torch.float32 or not bias.is_cuda:
            raise TypeError("bias must be a float32 CUDA tensor")
        bv = bias.expand(B, H, N, N)
        if bv.stride(3) != 1:
            raise ValueError("bias keys must be contiguous")
        rc = lib().attn_fwd_bias(_ptr(q), _ptr(k), _ptr(v), bv.data_ptr(), bv.stride(0),
                                 bv.stride(1), bv.stride(2), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                                 scale, int(bool(causal)), _dtype_code(q), _stream(stream))
    elif Hkv == H:
        rc = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, scale,
                            int(bool(causal)), _dtype_code(q), _stream(stream))
    else:
        rc = lib().attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                                scale, int(bool(causal)), _dtype_code(q), _stream(stream))
    _check(rc, "attn_fwd")
    return o, lse


def attn_fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False,
                    scale: float | None = None, out=None, lse=None, want_lse: bool = True,
                    stream=None):
    """Packed attention, q [T, H, d], k/v [T, H_kv, d], cu_seqlens int32
    [nseq+1] on the device -> (o [T,H,d], lse [H,T] fp32)."""
    _need_cuda(q, k, v, cu_seqlens)
    T, H, d = q.shape
    Hkv = k.shape[1]
    if cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    if k.shape != (T, Hkv, d) or v.shape != k.shape:
        raise ValueError("q [T,H,d] and k, v [T,H_kv,d] must agree in shape")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    if lse is None and want_lse:
        lse = torch.empty((H, T), device=q.device, dtype=torch.float32)
    _need_cuda(o, lse)
    if Hkv == H:
        rc = lib().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                   _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, int(max_seqlen),
                                   H, d, scale, int(bool(causal)), _dtype_code(q),
                                   _stream(stream))
    else:
        rc = lib().attn_fwd_varlen_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                       _ptr(cu_seqlens), cu_seqlens.numel() - 1, T,
                                       int(max_seqlen), H, Hkv, d, scale, int(bool(causal)),
                                       _dtype_code(q), _stream(stream))
    _check(rc, "attn_fwd_varlen")
    return o, lse


def attn_fwd_varlen_noalloc(q, k, v, cu_seqlens, max_seqlen: int, out, lse=None, status=None,
                            causal: bool = False, scale: float | None = None, stream=None):
    """attn_fwd_varlen for callers that cannot allocate device memory: the
    caller supplies every buffer (`out`, optional `lse` [H,T] fp32, optional
    one-element int32 `status` on the device) and the library uses only its
    fixed static scratch.  This wrapper allocates nothing either."""
    _need_cuda(q, k, v, cu_seqlens, out, lse, status)
    T, H, d = q.shape
    if cu_seqlens.dtype != torch.int32 or (status is not None and status.dtype != torch.int32):
        raise TypeError("cu_seqlens and status must be int32")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = lib().attn_fwd_varlen_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                       _ptr(cu_seqlens), cu_seqlens.numel() - 1, T,
                                       int(max_seqlen), H, d, scale, int(bool(causal)),
                                       _dtype_code(q), _ptr(status), _stream(stream))
    _check(rc, "attn_fwd_varlen_noalloc")
    return out, lse


def attn_fwd_paged(q, k_cache, v_cache, block_table, seqlens_k, max_seqlen_k: int,
                   causal: bool = True, scale: float | None = None, num_splits: int = 0,
                   out=None, lse=None, want_lse: bool = True, stream=None):
    """Decoding against a paged K/V cache: q [B, Nq, H, d] (the newest Nq
    positions), k_cache/v_cache [num_pages, page_size, H_kv, d], block_table
    int32 [B, max_pages], seqlens_k int32 [B] (all on the device)
    -> (o [B, Nq, H, d], lse [B, H, Nq] fp32)."""
    _need_cuda(q, k_cache, v_cache, block_table, seqlens_k)
    B, Nq, H, d = q.shape
    num_pages, page_size, Hkv, dk = k_cache.shape
    if v_cache.shape != k_cache.shape or dk != d or k_cache.dtype != q.dtype:
        raise ValueError("k_cache, v_cache must be [num_pages, page_size, H_kv, d] of q's dtype")
    if block_table.dtype != torch.int32 or seqlens_k.dtype != torch.int32:
        raise TypeError("block_table and seqlens_k must be int32")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    if lse is None and want_lse:
        lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    _need_cuda(o, lse)
    rc = lib().attn_fwd_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                              _ptr(seqlens_k), _ptr(o), _ptr(lse), B, Nq, H, Hkv, d, page_size,
                              block_table.shape[1], num_pages, int(max_seqlen_k), scale,
                              int(bool(causal)), _dtype_code(q), int(num_splits), _stream(stream))
    _check(rc, "attn_fwd_paged")
    return o, lse


def attn_bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None,
             stream=None):
    """Gradients of the dense forward: q, o, dout [B, N, H, d]; k, v
    [B, N, H_kv, d]; lse [B, H, N] fp32 from the forward -> (dq, dk, dv)."""
    _need_cuda(q, k, v, o, lse, dout)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc = lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                        _ptr(dk), _ptr(dv), B, H, Hkv, N, d, scale, int(bool(causal)),
                        _dtype_code(q), _stream(stream))
    _check(rc, "attn_bwd")
    return dq, dk, dv


def attn_fwd_host(q, k, v, causal: bool = False, scale: float | None = None, out=None,
                  lse=None, want_lse: bool = True, stream=None):
    """attn_fwd on HOST tensors q, k, v [B, N, H, d] (bf16/fp16, contiguous,
    page-locked for overlap) -> host (o, lse); the library pipelines the
    copies with the compute in chunks (batch entries, head groups of the
    first and last entry).  The call is asynchronous on `stream`:
    synchronise it before reading o and lse."""
    for t in (q, k, v, out, lse):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("attn_fwd_host takes contiguous host tensors")
    B, N, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    pin = q.is_pinned()
    o = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin) if out is None else out
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin)
    rc = lib().attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, scale,
                             int(bool(causal)), _dtype_code(q), _stream(stream))
    _check(rc, "attn_fwd_host")
    return o, lse


def attn_fwd_fp8_host(q, k, v, signs=None, causal: bool = False, scale: float | None = None,
                      out=None, lse=None, want_lse: bool = True, stream=None):
    """The 8-bit path on HOST tensors: bf16 q, k, v [B, N, H, d] (contiguous,
    page-locked for overlap), optional int8 signs [d] (host) -> host bf16 o
    and fp32 lse; block quantisation (with the rotation when signs are
    given) and the e4m3 forward run on the device per chunk, pipelined with
    the copies.  Asynchronous on `stream`: synchronise it before reading."""
    for t in (q, k, v, signs, out, lse):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("attn_fwd_fp8_host takes contiguous host tensors")
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("attn_fwd_fp8_host takes bf16 q, k, v")
    if signs is not None and (signs.dtype != torch.int8 or signs.numel() != q.shape[-1]):
        raise ValueError("signs must be int8 of length d")
    B, N, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    pin = q.is_pinned()
    o = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin) if out is None else out
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin)
    rc = lib().attn_fwd_fp8_host(_ptr(q), _ptr(k), _ptr(v), _ptr(signs), _ptr(o), _ptr(lse), B,
                                 H, N, d, scale, int(bool(causal)), _stream(stream))
    _check(rc, "attn_fwd_fp8_host")
    return o, lse


def attn_fwd_fp8(q8, k8, v8, descale_q, descale_k, descale_v, causal: bool = False,
                 scale: float | None = None, out=None, lse=None, want_lse: bool = True,
                 stream=None):
    """e4m3 attention: q8/k8/v8 [B,N,H,d] uint8 codes, descales fp32 [B,H,ceil(N/128)]
    -> (o [B,N,H,d] bf16, lse [B,H,N] fp32)."""
    _need_cuda(q8, k8, v8, descale_q, descale_k, descale_v)
    B, N, H, d = q8.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty(q8.shape, device=q8.device, dtype=torch.bfloat16) if out is None else out
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), device=q8.device, dtype=torch.float32)
    _need_cuda(o, lse)
    rc = lib().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(descale_q), _ptr(descale_k),
                            _ptr(descale_v), _ptr(o), _ptr(lse), B, H, N, d, scale,
                            int(bool(causal)), _stream(stream))
    _check(rc, "attn_fwd_fp8")
    return o, lse


def qkv_block_quant_hadamard(q, k, v, signs=None, per_tensor: bool = False, outs=None,
                             stream=None):
    """bf16 q/k/v [B,N,H,d] -> (q8, k8, v8 uint8 e4m3 codes, dq, dk, dv fp32 [B,H,nblk])."""
    _need_cuda(q, k, v, signs)
    B, N, H, d = q.shape
    nblk = (N + 127) // 128
    if outs is None:
        outs = [torch.empty(q.shape, device=q.device, dtype=torch.uint8) for _ in range(3)] + \
               [torch.empty((B, H, nblk), device=q.device, dtype=torch.float32) for _ in range(3)]
    q8, k8, v8, dq, dk, dv = outs
    rc = lib().qkv_block_quant_hadamard(_ptr(q), _ptr(k), _ptr(v), _ptr(q8), _ptr(k8),
                                        _ptr(v8), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(signs),
                                        int(bool(per_tensor)), B, H, N, d, _stream(stream))
    _check(rc, "qkv_block_quant_hadamard")
    return q8, k8, v8, dq, dk, dv


def get_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status word (0 = ok)."""
    return int(lib().attn_get_status(_stream(stream)))


def check_status(stream=None):
    _check(get_status(stream), "device")
