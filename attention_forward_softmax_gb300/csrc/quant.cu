// quant.cu -- fp8 pre-step: incoherent processing and block quantisation
// ("Fused attention kernel", wikillm concept card, section "8-bit forward
// pass (FP8, Hopper)": one scale per block of Q, K and V; Q and K multiplied
// by a random-sign diagonal times a Hadamard matrix before quantisation).
//
// Persistent CTAs of 4 warps (two per SM) walk the (tensor, batch, head,
// 128-token block) items.  Each item's 128 x d bf16 rows arrive in shared
// memory by TMA (128-byte swizzle, so a warp reading 32 rows at once meets
// no bank conflict), double-buffered so the next item's copy streams while
// this one is processed.  One thread holds one token row: for Q and K it
// flips the signs on the packed bf16 pairs (x * diag(s)), then runs the whole
// d-point fast Walsh-Hadamard transform in its registers -- the stride-1
// stage on scalars, the others as packed f32x2 add/sub -- which equals
// x * diag(s) * H_d with H_d the Sylvester matrix; the 1/sqrt(d) is folded
// into the quantisation multiplier.  The block's amax is combined across the
// four warps through shared memory, scale = amax / 448, and every value is
// multiplied by 1/scale and rounded to e4m3 (nearest even, saturating).  The
// codes go to a swizzled shared-memory tile that one TMA store writes back.
// HBM-bound: 2 bytes read and 1 byte written per element.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

namespace {

constexpr int kQThreads = 128;   // one 128-token block per item, one row per thread

struct QuantArgs {
  float *descale[3];
  const int8_t *signs;   // may be null
  int B, H, N, nblk;
  int mode;              // 0: block scales; 1: amax only (per-tensor pass 1); 2: quantise with
                         //    the per-tensor scale in tensor_amax (pass 2)
  const float *tensor_amax;  // [3], mode 2
  int *status;
  long long budget;
};

// Shared memory of one CTA (offsets from a 1024-byte aligned base).
template <int D>
struct QuantSmem {
  static constexpr int kInBytes = 128 * D * 2;    // one block of bf16 rows: D / 64 chunks of
                                                  // 128 rows x 128 bytes
  static constexpr int kOutBytes = 128 * D;       // one block of e4m3 codes
  static constexpr int kOffOut = 2 * kInBytes;
  static constexpr int kOffMask = kOffOut + 2 * kOutBytes;
  static constexpr int kBytes = kOffMask + D / 2 * 4 + 1024;
};

// Byte offset of 16-byte unit u of row r in a tile of rows of D codes, as
// the tensor copy swizzles it (128-byte rows: unit ^ (row mod 8); 64-byte
// rows: unit ^ ((row / 2) mod 4)).
template <int D>
__device__ __forceinline__ uint32_t code_unit(int r, int u) {
  if constexpr (D == 128)
    return r * 128 + ((u ^ (r & 7)) << 4);
  else
    return r * 64 + ((u ^ ((r >> 1) & 3)) << 4);
}

template <int D>
__global__ void __launch_bounds__(kQThreads, 2)
    quant_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap yq,
                 const __grid_constant__ CUtensorMap yk, const __grid_constant__ CUtensorMap yv,
                 const QuantArgs a) {
  using L = QuantSmem<D>;
  constexpr int NP = D / 2;              // channel pairs of a row
  extern __shared__ uint8_t qsm_raw[];
  uint8_t *qsm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(qsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *in = qsm;
  uint8_t *out = qsm + L::kOffOut;
  uint32_t *smask = reinterpret_cast<uint32_t *>(qsm + L::kOffMask);
  __shared__ uint64_t full[2];
  __shared__ float red[kQThreads / 32];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = threadIdx.x;             // the row of each block this thread processes
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
    tma_prefetch_desc(&yq);
    tma_prefetch_desc(&yk);
    tma_prefetch_desc(&yv);
  }
  // sign diagonal as XOR masks on bf16 pairs: bit 15 flips channel 2i,
  // bit 31 channel 2i + 1
  for (int i = threadIdx.x; i < NP; i += kQThreads)
    smask[i] = a.signs == nullptr ? 0u
                                  : ((a.signs[2 * i] < 0 ? 0x8000u : 0u) |
                                     (a.signs[2 * i + 1] < 0 ? 0x80000000u : 0u));
  __syncthreads();
  const WaitCtl wc{&abort_flag, a.status, a.budget};

  // item -> (tensor, b, h, blk), blocks of one (b, h) consecutive
  auto issue = [&](int it, int buf) {
    const int tensor = it / bhn, rem = it % bhn;
    const int bh = rem / a.nblk, blk = rem % a.nblk;
    const CUtensorMap *m = tensor == 0 ? &mq : (tensor == 1 ? &mk : &mv);
    mbar_arrive_expect_tx(&full[buf], L::kInBytes);
#pragma unroll
    for (int c = 0; c < D / 64; ++c)
      tma_load_4d(in + buf * L::kInBytes + c * 16384, m, &full[buf], c * 64, bh % a.H, blk * 128,
                  bh / a.H);
  };
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
    // reading it before the previous item's amax barrier.
    const int nxt = it + gridDim.x;
    if (nxt < items) {
      if (threadIdx.x == 0) {
        fence_proxy_async_smem();
        issue(nxt, buf ^ 1);
      }
      ++issued[buf ^ 1];
    }
    // the code tile of two items ago must have been read by its store
    if (threadIdx.x == 0) bulk_wait_group_read<1>();
    // every thread leaves together if any wait gave up
    const bool got = mbar_wait(&full[buf], waited[buf] & 1, wc);
    if (!named_bar_and(1, kQThreads, got)) { ok = false; break; }
    ++waited[buf];

    const int tensor = it / bhn, rem = it % bhn;
    const int bh = rem / a.nblk, blk = rem % a.nblk;
    const int b = bh / a.H, h = bh % a.H;
    const bool rotate = (tensor < 2) && (a.signs != nullptr);

    // this thread's row, as channel pairs (2i, 2i + 1) of fp32
    uint64_t v[NP];
    const uint8_t *rowp = in + buf * L::kInBytes + r * 128;
#pragma unroll
    for (int c = 0; c < D / 64; ++c)
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(rowp + c * 16384 + ((u ^ (r & 7)) << 4));
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = c * 32 + u * 4 + q;
          const uint32_t x = rotate ? w[q] ^ smask[i] : w[q];
          v[i] = f32x2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
        }
      }
    if (rotate) {
      // channel stride 1: the two halves of each pair
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        float lo, hi;
        f32x2_split(v[i], lo, hi);
        v[i] = f32x2(lo + hi, lo - hi);
      }
      // channel strides 2 .. D/2: pairs hs apart
#pragma unroll
      for (int hs = 1; hs < NP; hs <<= 1)
#pragma unroll
        for (int i = 0; i < NP; ++i)
          if ((i & hs) == 0) {
            const uint64_t x0 = v[i], x1 = v[i + hs];
            v[i] = add_f32x2(x0, x1);
            v[i + hs] = sub_f32x2(x0, x1);
          }
    }
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      float lo, hi;
      f32x2_split(v[i], lo, hi);
      am = fmax3(am, fabsf(lo), fabsf(hi));
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, m));
    if (lane == 0) red[warp] = am;
    named_bar_sync(2, kQThreads);
    float bmax = red[0];
#pragma unroll
    for (int w = 1; w < kQThreads / 32; ++w) bmax = fmaxf(bmax, red[w]);
    const float norm = rotate ? 1.f / sqrtf(static_cast<float>(D)) : 1.f;
    const float amax = bmax * norm;          // of the rotated (orthonormal) values

    float *dsc = tensor == 0 ? a.descale[0] : (tensor == 1 ? a.descale[1] : a.descale[2]);
    const size_t dslot = (static_cast<size_t>(b) * a.H + h) * a.nblk + blk;
    if (a.mode == 1) {
      if (threadIdx.x == 0) dsc[dslot] = amax;
      continue;
    }
    const float amx = (a.mode == 2) ? a.tensor_amax[tensor] : amax;
    const float scale = amx > 0.f ? amx / 448.f : 1.f;
    const float mul = norm * (1.f / scale);  // codes from x * (1/scale), see the header
    if (threadIdx.x == 0) dsc[dslot] = scale;
    const uint64_t mul2 = f32x2(mul, mul);
    uint8_t *tile = out + buf * L::kOutBytes;
#pragma unroll
    for (int u = 0; u < D / 16; ++u) {       // 16 codes = 8 pairs per 16-byte unit
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float x0, x1, x2, x3;
        f32x2_split(mul_f32x2(v[8 * u + 2 * q], mul2), x0, x1);
        f32x2_split(mul_f32x2(v[8 * u + 2 * q + 1], mul2), x2, x3);
        w[q] = pack_e4m3x4(x0, x1, x2, x3);
      }
      st_shared_v4(smem_addr(tile) + code_unit<D>(r, u), w[0], w[1], w[2], w[3]);
    }
    fence_proxy_async_smem();                // codes visible to the tensor store
    named_bar_sync(3, kQThreads);
    if (threadIdx.x == 0) {
      const CUtensorMap *y = tensor == 0 ? &yq : (tensor == 1 ? &yk : &yv);
      tma_store_4d(y, tile, 0, h, blk * 128, b);   // rows past N are not written
      bulk_commit_group();
    }
  }
  if (threadIdx.x == 0) {
    // After a wait gave up: let every copy this CTA started land before exit.
    if (!ok)
      for (int b2 = 0; b2 < 2; ++b2)
        for (int k2 = waited[b2]; k2 < issued[b2]; ++k2) mbar_wait_drain(&full[b2], k2 & 1);
    bulk_wait_group_read<0>();               // shared memory stays until the stores read it
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
  // Inputs: one 128-token block of one (b, h) per item, as d / 64 copies of
  // a (64, 1, 128, 1) box of the (d, H, N, B) bf16 tensor with the 128-byte
  // swizzle; rows past N are zero-filled.  Outputs: a (d, 1, 128, 1) box of
  // the (d, H, N, B) code tensor, swizzled to match; rows past N are not
  // written.
  CUtensorMap maps[6];
  const void *src[3] = {q, k, v};
  void *dst[3] = {q8, k8, v8};
  for (int t = 0; t < 3; ++t) {
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2,
                                   (cuuint64_t)N * H * d * 2};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    if ((st = encode_tiled(&maps[t], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, src[t], dims, strides,
                           box, CU_TENSOR_MAP_SWIZZLE_128B)) != ATTN_OK)
      return st;
    const cuuint64_t ystrides[3] = {(cuuint64_t)d, (cuuint64_t)H * d, (cuuint64_t)N * H * d};
    const cuuint32_t ybox[4] = {(cuuint32_t)d, 1, 128, 1};
    if ((st = encode_tiled(&maps[3 + t], CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, dst[t], dims, ystrides,
                           ybox, d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B)) !=
        ATTN_OK)
      return st;
  }
  QuantArgs a{};
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
                                                  QuantSmem<128>::kBytes)
                           : cudaFuncSetAttribute(quant_kernel<64>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  QuantSmem<64>::kBytes);
  });
  if (attr_err[di][dev] != cudaSuccess) return ATTN_ERR_LAUNCH;
  auto run = [&](int mode) {
    a.mode = mode;
    if (d == 128)
      quant_kernel<128><<<grid, kQThreads, QuantSmem<128>::kBytes, s>>>(
          maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], a);
    else
      quant_kernel<64><<<grid, kQThreads, QuantSmem<64>::kBytes, s>>>(
          maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], a);
    return cudaGetLastError() == cudaSuccess;
  };
  if (!per_tensor) return run(0) ? ATTN_OK : ATTN_ERR_LAUNCH;
  if (!run(1)) return ATTN_ERR_LAUNCH;
  tensor_amax_kernel<<<3, 1024, 0, s>>>(descale_q, descale_k, descale_v,
                                        static_cast<int>(B * H * nblk), ds->scratch_amax);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  return run(2) ? ATTN_OK : ATTN_ERR_LAUNCH;
}
