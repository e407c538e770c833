// quant.cu -- fp8 pre-step: incoherent processing and block quantisation
// ("Fused attention kernel", wikillm concept card, section "8-bit forward
// pass (FP8, Hopper)": one scale per block of Q, K and V; Q and K multiplied
// by a random-sign diagonal times a Hadamard matrix before quantisation).
//
// Persistent CTAs (two per SM, 16 warps each) walk the (tensor, batch, head,
// 128-token block) items.  Each item's 128 x d bf16 rows arrive in shared
// memory by one TMA copy, issued while the previous item is being processed
// (two buffers), so HBM reads stream continuously.  A token row of d channels
// is spread over 8 lanes (d/8 consecutive channels per lane), so a warp holds
// 4 rows at a time and each warp owns 8 rows of the block.  For Q and K the
// row is multiplied by the signs, then transformed by a fast Walsh-Hadamard
// transform -- butterflies inside a lane for the small strides, then across
// the 8 lanes with shuffles (one shuffle and one fused multiply-add with a +-1
// sign per element and stage) -- then scaled by 1/sqrt(d); this equals
// x * diag(s) * H_d / sqrt(d) with H_d the Sylvester matrix.  The block's amax
// is reduced through shared memory, scale = amax / 448, and every value is
// multiplied by 1/scale and rounded to e4m3 (nearest even, saturating).
// HBM-bound: 2 bytes read and 1 byte written per element.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

namespace {

constexpr int kQThreads = 512;
constexpr int kLanesPerRow = 8;
constexpr int kRowsPerPass = 32 / kLanesPerRow;          // rows a warp holds at once
constexpr int kPasses = 128 / (kQThreads / 32) / kRowsPerPass;   // 2

struct QuantArgs {
  uint8_t *y[3];
  float *descale[3];
  const int8_t *signs;   // may be null
  int B, H, N, nblk;
  int mode;              // 0: block scales; 1: amax only (per-tensor pass 1); 2: quantise with
                         //    the per-tensor scale in tensor_amax (pass 2)
  const float *tensor_amax;  // [3], mode 2
  int *status;
  long long budget;
};

template <int D>
constexpr int quant_smem_bytes() { return 2 * 128 * D * 2 + 1024; }

template <int D>
__global__ void __launch_bounds__(kQThreads, 2)
    quant_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mv, const QuantArgs a) {
  constexpr int EPL = D / kLanesPerRow;   // channels per lane: 16 (d=128) or 8 (d=64)
  constexpr int kBufBytes = 128 * D * 2;
  extern __shared__ uint8_t qsm_raw[];
  uint8_t *qsm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(qsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t full[2];
  __shared__ float red[2][kQThreads / 32];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow;     // row within a pass
  const int gl = lane % kLanesPerRow;      // lane within the row's group
  const int bhn = a.B * a.H * a.nblk;
  const int items = 3 * bhn;
  if (threadIdx.x == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&mq);
    tma_prefetch_desc(&mk);
    tma_prefetch_desc(&mv);
  }
  __syncthreads();
  const WaitCtl wc{&abort_flag, a.status, a.budget};

  // item -> (tensor, b, h, blk), blocks of one (b, h) consecutive
  auto issue = [&](int it, int buf) {
    const int tensor = it / bhn, rem = it % bhn;
    const int bh = rem / a.nblk, blk = rem % a.nblk;
    const CUtensorMap *m = tensor == 0 ? &mq : (tensor == 1 ? &mk : &mv);
    mbar_arrive_expect_tx(&full[buf], kBufBytes);
    tma_load_4d(qsm + buf * kBufBytes, m, &full[buf], 0, bh % a.H, blk * 128, bh / a.H);
  };
  // sign diagonal as a bit mask (bit e: channel gl*EPL+e is negated)
  uint32_t sgn_bits = 0;
  if (a.signs != nullptr)
#pragma unroll
    for (int e = 0; e < EPL; ++e) sgn_bits |= (a.signs[gl * EPL + e] < 0 ? 1u : 0u) << e;
  int issued[2] = {0, 0}, waited[2] = {0, 0};
  int it = blockIdx.x;
  if (it < items) {
    if (threadIdx.x == 0) issue(it, 0);
    issued[0] = 1;
  }
  bool ok = true;
  for (int kk = 0; it < items; it += gridDim.x, ++kk) {
    const int buf = kk & 1;
    // Prefetch the next item into the other buffer: every thread finished
    // reading that buffer before the previous item's barrier.
    const int nxt = it + gridDim.x;
    if (nxt < items) {
      if (threadIdx.x == 0) {
        fence_proxy_async_smem();
        issue(nxt, buf ^ 1);
      }
      ++issued[buf ^ 1];
    }
    // every thread leaves together if any wait gave up (no thread is left at
    // the block barrier below)
    const bool got = mbar_wait(&full[buf], waited[buf] & 1, wc);
    if (!__syncthreads_and(got)) { ok = false; break; }
    ++waited[buf];

    const int tensor = it / bhn, rem = it % bhn;
    const int bh = rem / a.nblk, blk = rem % a.nblk;
    const int b = bh / a.H, h = bh % a.H;
    const bool rotate = (tensor < 2) && (a.signs != nullptr);
    float *dsc = tensor == 0 ? a.descale[0] : (tensor == 1 ? a.descale[1] : a.descale[2]);
    uint8_t *yout = tensor == 0 ? a.y[0] : (tensor == 1 ? a.y[1] : a.y[2]);

    float v[kPasses][EPL];
    int tok[kPasses];
    const uint8_t *src = qsm + buf * kBufBytes;
#pragma unroll
    for (int r = 0; r < kPasses; ++r) {
      const int row = (warp * kPasses + r) * kRowsPerPass + sub;   // row within the block
      tok[r] = blk * 128 + row;
      // rows past N arrive zero-filled from the copy
#pragma unroll
      for (int q = 0; q < EPL / 8; ++q) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(src + (row * D + gl * EPL + q * 8) * 2);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162 *>(&w[u]);
          v[r][q * 8 + 2 * u] = __low2float(p2);
          v[r][q * 8 + 2 * u + 1] = __high2float(p2);
        }
      }
    }
    if (rotate) {
      const float norm = 1.f / sqrtf(static_cast<float>(D));
#pragma unroll
      for (int r = 0; r < kPasses; ++r) {
#pragma unroll
        for (int e = 0; e < EPL; ++e)
          v[r][e] = __uint_as_float(__float_as_uint(v[r][e]) ^ (((sgn_bits >> e) & 1u) << 31));
        // butterflies between channels of one lane (strides 1, 2, 4, ...)
#pragma unroll
        for (int hs = 1; hs < EPL; hs <<= 1)
#pragma unroll
          for (int e = 0; e < EPL; ++e)
            if ((e & hs) == 0) {
              const float u = v[r][e], w = v[r][e + hs];
              v[r][e] = u + w;
              v[r][e + hs] = u - w;
            }
        // butterflies across the row's lanes (channel stride EPL * m): the
        // lane holding the upper channel keeps other - mine, the lower
        // mine + other
#pragma unroll
        for (int m = 1; m < kLanesPerRow; m <<= 1) {
          const float sgn = (gl & m) ? -1.f : 1.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) {
            const float other = __shfl_xor_sync(0xffffffffu, v[r][e], m);
            v[r][e] = fmaf(v[r][e], sgn, other);
          }
        }
#pragma unroll
        for (int e = 0; e < EPL; ++e) v[r][e] *= norm;
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int r = 0; r < kPasses; ++r)
#pragma unroll
      for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(v[r][e]));
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    // red is double-buffered: a thread can be one item ahead of the slowest
    if (lane == 0) red[kk & 1][warp] = amax;
    __syncthreads();
    float bmax = 0.f;
#pragma unroll
    for (int w = 0; w < kQThreads / 32; ++w) bmax = fmaxf(bmax, red[kk & 1][w]);

    const size_t dslot = (static_cast<size_t>(b) * a.H + h) * a.nblk + blk;
    if (a.mode == 1) {
      if (threadIdx.x == 0) dsc[dslot] = bmax;
      continue;
    }
    const float amx = (a.mode == 2) ? a.tensor_amax[tensor] : bmax;
    const float scale = amx > 0.f ? amx / 448.f : 1.f;
    const float inv = 1.f / scale;   // codes from x * (1/scale): within 2 ulp of x / scale
    if (threadIdx.x == 0) dsc[dslot] = scale;
#pragma unroll
    for (int r = 0; r < kPasses; ++r) {
      if (tok[r] >= a.N) continue;
      const size_t off = ((static_cast<size_t>(b) * a.N + tok[r]) * a.H + h) * D + gl * EPL;
      uint32_t w[EPL / 4];
#pragma unroll
      for (int q = 0; q < EPL / 4; ++q)
        w[q] = pack_e4m3x4(v[r][4 * q] * inv, v[r][4 * q + 1] * inv, v[r][4 * q + 2] * inv,
                           v[r][4 * q + 3] * inv);
      if constexpr (EPL == 16)
        *reinterpret_cast<uint4 *>(yout + off) = make_uint4(w[0], w[1], w[2], w[3]);
      else
        *reinterpret_cast<uint2 *>(yout + off) = make_uint2(w[0], w[1]);
    }
  }
  // After a wait gave up: let every copy this CTA started land before exit.
  if (!ok && threadIdx.x == 0) {
    for (int b2 = 0; b2 < 2; ++b2)
      for (int k2 = waited[b2]; k2 < issued[b2]; ++k2) mbar_wait_drain(&full[b2], k2 & 1);
  }
}

// Per-tensor pass between the two quantisation passes: max over the block
// amaxes of each tensor.
__global__ void tensor_amax_kernel(const float *dq, const float *dk, const float *dv, int n,
                                   float *out) {
  const float *src = blockIdx.x == 0 ? dq : (blockIdx.x == 1 ? dk : dv);
  float m = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, src[i]);
  __shared__ float red[32];
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r = fmaxf(r, red[w]);
    out[blockIdx.x] = r;
  }
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" attn_status_t qkv_block_quant_hadamard(const void *q, const void *k, const void *v,
                                                  void *q8, void *k8, void *v8,
                                                  float *descale_q, float *descale_k,
                                                  float *descale_v, const int8_t *signs,
                                                  int per_tensor, int B, int H, int N, int d,
                                                  void *stream) {
  if (!q || !k || !v || !q8 || !k8 || !v8 || !descale_q || !descale_k || !descale_v)
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q8) || !aligned16(k8) ||
      !aligned16(v8))
    return ATTN_ERR_MISALIGNED;
  const long long nblk = (N + 127) / 128;
  if (static_cast<long long>(B) * H > 65535 || nblk > 0x7fffffff ||
      static_cast<long long>(B) * N * H * d > (1LL << 40))
    return ATTN_ERR_TOO_LARGE;
  DeviceState *ds = nullptr;
  attn_status_t st = device_state(&ds);
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // one 128-token block of one (b, h) per copy: box (d, 1, 128, 1) of the
  // (d, H, N, B) bf16 tensor, rows past N zero-filled
  CUtensorMap maps[3];
  const void *src[3] = {q, k, v};
  for (int t = 0; t < 3; ++t) {
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2,
                                   (cuuint64_t)N * H * d * 2};
    const cuuint32_t box[4] = {(cuuint32_t)d, 1, 128, 1};
    if ((st = encode_tiled(&maps[t], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, src[t], dims, strides,
                           box, CU_TENSOR_MAP_SWIZZLE_NONE)) != ATTN_OK)
      return st;
  }
  QuantArgs a{};
  a.y[0] = static_cast<uint8_t *>(q8);
  a.y[1] = static_cast<uint8_t *>(k8);
  a.y[2] = static_cast<uint8_t *>(v8);
  a.descale[0] = descale_q;
  a.descale[1] = descale_k;
  a.descale[2] = descale_v;
  a.signs = signs;
  a.B = B; a.H = H; a.N = N; a.nblk = static_cast<int>(nblk);
  a.tensor_amax = ds->scratch_amax;
  a.status = ds->status;
  a.budget = wait_budget();
  const long long items = 3LL * B * H * nblk;
  const int grid = static_cast<int>(std::min<long long>(items, 2LL * ds->num_sms));
  // shared-memory attribute: once per device and head dimension (call_once
  // serialises concurrent first calls)
  static std::once_flag attr_once[2][kMaxDevices];
  static cudaError_t attr_err[2][kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  const int di = d == 128 ? 1 : 0;
  std::call_once(attr_once[di][dev], [di, dev] {
    attr_err[di][dev] = di ? cudaFuncSetAttribute(quant_kernel<128>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  quant_smem_bytes<128>())
                           : cudaFuncSetAttribute(quant_kernel<64>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  quant_smem_bytes<64>());
  });
  if (attr_err[di][dev] != cudaSuccess) return ATTN_ERR_LAUNCH;
  auto run = [&](int mode) {
    a.mode = mode;
    if (d == 128)
      quant_kernel<128><<<grid, kQThreads, quant_smem_bytes<128>(), s>>>(maps[0], maps[1], maps[2], a);
    else
      quant_kernel<64><<<grid, kQThreads, quant_smem_bytes<64>(), s>>>(maps[0], maps[1], maps[2], a);
    return cudaGetLastError() == cudaSuccess;
  };
  if (!per_tensor) return run(0) ? ATTN_OK : ATTN_ERR_LAUNCH;
  if (!run(1)) return ATTN_ERR_LAUNCH;
  tensor_amax_kernel<<<3, 1024, 0, s>>>(descale_q, descale_k, descale_v,
                                        static_cast<int>(B * H * nblk), ds->scratch_amax);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  return run(2) ? ATTN_OK : ATTN_ERR_LAUNCH;
}
