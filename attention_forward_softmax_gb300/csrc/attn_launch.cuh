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
    const cuuint64_t dims[3] = {(cuuint64_t)a.d, (cuuint64_t)heads, (cuuint64_t)a.T};
    const cuuint64_t strides[2] = {a.d * e, (cuuint64_t)heads * a.d * e};
    const cuuint32_t box[3] = {(cuuint32_t)C::kChunkElems, 1, 128};
    return encode_tiled(m, tma_dtype<C>(), 3, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    const cuuint64_t dims[4] = {(cuuint64_t)a.d, (cuuint64_t)heads, (cuuint64_t)a.N,
                                (cuuint64_t)a.B};
    const cuuint64_t strides[3] = {a.d * e, (cuuint64_t)heads * a.d * e,
                                   (cuuint64_t)a.N * heads * a.d * e};
    const cuuint32_t box[4] = {(cuuint32_t)C::kChunkElems, 1, 128, 1};
    return encode_tiled(m, tma_dtype<C>(), 4, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
}

// Combines the two key halves of each split tile (the running-softmax merge
// over disjoint key sets): lse = log(e^lse0 + e^lse1), O = e^(lse0 - lse) O0
// + e^(lse1 - lse) O1, rounded to the output type.  One warp per row.
template <int D, bool F16Out>
__global__ void __launch_bounds__(256) split_merge_kernel(const float *part_o, const float *part_lse,
                                                          void *o, float *lse, int first_tile,
                                                          int rem, int nqt, int H, int N) {
  const int w = (blockIdx.x * 256 + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int sidx = w >> 8, r = w & 255;
  if (sidx >= rem) return;
  const int t = first_tile + sidx, bh = t / nqt, b = bh / H, h = bh % H;
  const int row = (t % nqt) * 256 + r;
  if (row >= N) return;
  const size_t p0 = (static_cast<size_t>(2 * sidx) * 256 + r), p1 = p0 + 256;
  const float l0 = part_lse[p0], l1 = part_lse[p1];
  const float m = fmaxf(l0, l1);
  const float e0 = expf(l0 - m), e1 = expf(l1 - m);
  const float inv = 1.f / (e0 + e1);
  const float w0 = e0 * inv, w1 = e1 * inv;
  constexpr int kPer = D / 32;                       // 4 (d = 128) or 2 (d = 64)
  const float *a0 = part_o + p0 * D + lane * kPer, *a1 = part_o + p1 * D + lane * kPer;
  float v[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) v[i] = w0 * a0[i] + w1 * a1[i];
  uint32_t wd[kPer / 2];
#pragma unroll
  for (int i = 0; i < kPer / 2; ++i)
    wd[i] = F16Out ? pack_f16(v[2 * i], v[2 * i + 1]) : pack_bf16(v[2 * i], v[2 * i + 1]);
  uint16_t *orow = static_cast<uint16_t *>(o) + ((static_cast<size_t>(b) * N + row) * H + h) * D;
  if constexpr (kPer == 4)
    *reinterpret_cast<uint2 *>(orow + lane * 4) = make_uint2(wd[0], wd[1]);
  else
    *reinterpret_cast<uint32_t *>(orow + lane * 2) = wd[0];
  if (lane == 0 && lse != nullptr)
    lse[(static_cast<size_t>(b) * H + h) * N + row] = m + logf(e0 + e1);
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
  p.d_out = a.d;
  p.wait_budget = a.budget;
  p.status = a.status;
  p.bias = a.bias;
  p.bias_sb = a.bias_sb;
  p.bias_sh = a.bias_sh;
  p.bias_sr = a.bias_sr;
  // dense, non-causal: the last split_rem tiles run as two key halves each
  const int split_rem = C::kVarlen ? 0 : a.split_rem;
  p.split_from = split_rem > 0 ? a.num_tiles - split_rem : -1;
  p.part_o = a.part_o;
  p.part_lse = a.part_lse;
  p.num_tiles = a.num_tiles + split_rem;
  const int grid = p.num_tiles < a.num_sms ? p.num_tiles : a.num_sms;
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
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  if (split_rem > 0) {
    const unsigned blocks = static_cast<unsigned>((static_cast<size_t>(split_rem) * 256 * 32 + 255) / 256);
    split_merge_kernel<C::D, C::E == Elem::F16><<<blocks, 256, 0, s>>>(
        a.part_o, a.part_lse, a.o, a.lse, p.split_from, split_rem, (a.N + 255) / 256, a.H, a.N);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

}  // namespace attn
