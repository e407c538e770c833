// attn_launch.cuh -- host launcher for one kernel instantiation: builds the
// Q/K/V tensor maps (128-byte swizzle, 128-row boxes) and launches a
// persistent grid of at most one CTA per SM on the caller's stream.
#pragma once

#include <mutex>

#include "attn_kernel.cuh"
#include "internal.h"

namespace attn {

template <class C>
CUtensorMapDataType tma_dtype() {
  if constexpr (C::E == Elem::BF16) return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  else if constexpr (C::E == Elem::F16) return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  else return CU_TENSOR_MAP_DATA_TYPE_UINT8;
}

// Tensor map of Q (heads = H) or K / V (heads = H_kv).
template <class C>
attn_status_t make_qkv_map(CUtensorMap *m, const void *ptr, const LaunchArgs &a, int heads) {
  const cuuint64_t e = C::kElt;
  if constexpr (C::kVarlen) {
    const cuuint64_t dims[3] = {(cuuint64_t)C::D, (cuuint64_t)heads, (cuuint64_t)a.T};
    const cuuint64_t strides[2] = {C::D * e, (cuuint64_t)heads * C::D * e};
    const cuuint32_t box[3] = {(cuuint32_t)C::kChunkElems, 1, 128};
    return encode_tiled(m, tma_dtype<C>(), 3, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    const cuuint64_t dims[4] = {(cuuint64_t)C::D, (cuuint64_t)heads, (cuuint64_t)a.N,
                                (cuuint64_t)a.B};
    const cuuint64_t strides[3] = {C::D * e, (cuuint64_t)heads * C::D * e,
                                   (cuuint64_t)a.N * heads * C::D * e};
    const cuuint32_t box[4] = {(cuuint32_t)C::kChunkElems, 1, 128, 1};
    return encode_tiled(m, tma_dtype<C>(), 4, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
}

template <class C>
attn_status_t launch_cfg(const LaunchArgs &a, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  attn_status_t st;
  if ((st = make_qkv_map<C>(&mq, a.q, a, a.H)) != ATTN_OK) return st;
  if ((st = make_qkv_map<C>(&mk, a.k, a, a.Hkv)) != ATTN_OK) return st;
  if ((st = make_qkv_map<C>(&mv, a.v, a, a.Hkv)) != ATTN_OK) return st;
  Params p{};
  p.o = a.o;
  p.lse = a.lse;
  p.cu_seqlens = a.cu_seqlens;
  p.tiles = a.tiles;
  p.num_entries = a.num_entries;
  p.B = a.B;
  p.H = a.H;
  p.grp = a.H / a.Hkv;
  p.N = a.N;
  p.T = a.T;
  p.num_tiles = a.num_tiles;
  p.causal = a.causal;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.dq = a.dq;
  p.dk = a.dk;
  p.dv = a.dv;
  p.nblk = (a.N + 127) / 128;
  p.wait_budget = a.budget;
  p.status = a.status;
  p.bias = a.bias;
  p.bias_sb = a.bias_sb;
  p.bias_sh = a.bias_sh;
  p.bias_sr = a.bias_sr;
  const int grid = a.num_tiles < a.num_sms ? a.num_tiles : a.num_sms;
  if (grid <= 0) return ATTN_OK;
  // The shared-memory attribute is set once per device and instantiation;
  // concurrent first calls from several host threads are serialised by
  // call_once.
  static std::once_flag attr_once[kMaxDevices];
  static cudaError_t attr_err[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::call_once(attr_once[dev], [dev] {
    attr_err[dev] = cudaFuncSetAttribute(attn_fwd_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
  });
  if (attr_err[dev] != cudaSuccess) return ATTN_ERR_LAUNCH;
  attn_fwd_kernel<C><<<grid, C::kThreads, C::kSmemBytes, s>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace attn
