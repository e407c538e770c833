// bwd.cu -- backward pass of the fused attention: dQ, dK, dV from Q, K, V,
// the forward's O and lse, and the upstream gradient dO (the backward pass
// of the FlashAttention-3 summary, arxivlens, Key Results, and of the
// "Fused attention kernel" card, "When to use which").
//
// With S = scale Q K^T over the allowed keys, P = exp(S - lse) (the forward's
// softmax, recomputed from its lse), D_i = rowsum(dO_i * O_i):
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  dQ = scale dS K,
//   dK = scale dS^T Q;
// grouped K/V heads sum dK and dV over their query heads.
//
// Layout on the GPU (d = 128, 16-bit):
//  * one CTA per (batch, K/V head, 128-key block); it loops over the query
//    heads of its group and their 64-row query blocks (causal: the blocks at
//    or after its keys).  dK and dV accumulate in TMEM for the whole loop;
//  * per query block, five tcgen05 MMAs: S^T = K Q^T and dP^T = V dO^T (both
//    operands K-major), then -- after the four softmax warps (one thread per
//    key row) have turned them into P^T and dS^T in shared memory -- dV +=
//    P^T dO and dK += dS^T Q (dO and Q read MN-major, as V in the forward),
//    and dQ^T = K^T dS^T (K read MN-major as the A operand);
//  * dQ^T leaves TMEM through the softmax warps (one thread per head-dim
//    column) into an fp32 accumulator in global memory by atomic adds; a last
//    pass scales it and rounds it to the output type;
//  * TMEM: S^T [0,64), dP^T [64,128), dV [128,256), dK [256,384), dQ^T
//    [384,448);
//  * every mbarrier wait is bounded; on expiry the status word gets
//    ATTN_ERR_TIMEOUT and the CTA drains its copies and MMAs and returns.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_kernel.cuh"
#include "internal.h"

namespace attn {
namespace {

constexpr int kBwdD = 128;
constexpr int kBC = 128;                    // keys per CTA
constexpr int kBR = 64;                     // query rows per block
constexpr int kBwdThreads = 192;            // 4 softmax warps, MMA warp, TMA warp
constexpr int kWarpMMAb = 4, kWarpTMAb = 5;

struct BwdParams {
  const float *lse;                         // [B, H, N] natural log
  const float *Dvec;                        // [B, H, N] rowsum(dO * O)
  float *dq_acc;                            // [B, N, H, d] fp32, zeroed
  void *dk, *dv;                            // [B, N, H_kv, d]
  int B, H, Hkv, N;
  float scale, scale_log2;
  int causal;
  long long wait_budget;
  int *status;
};

struct BwdSmem {
  static constexpr int kKVBytes = kBC * kBwdD * 2;        // 32 KB: 2 chunks of 128 rows x 128 B
  static constexpr int kQBytes = kBR * kBwdD * 2;         // 16 KB: 2 chunks of 64 rows x 128 B
  static constexpr int kPBytes = kBC * kBR * 2;           // 16 KB: 128 rows x 128 B
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKVBytes;
  static constexpr int kOffQ = kOffV + kKVBytes;          // [2 buffers]
  static constexpr int kOffDO = kOffQ + 2 * kQBytes;      // [2 buffers]
  static constexpr int kOffP = kOffDO + 2 * kQBytes;
  static constexpr int kOffDS = kOffP + kPBytes;
  static constexpr int kOffBar = kOffDS + kPBytes;
  static constexpr int kNumBars = 12;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 64 + 1024;     // + alignment slack
};

constexpr uint32_t kColS = 0, kColDP = 64, kColDV = 128, kColDK = 256, kColDQ = 384;

template <Elem E>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ BwdParams p) {
  using L = BwdSmem;
  constexpr uint32_t kFmt = (E == Elem::BF16) ? 1u : 0u;
  constexpr uint32_t kIdS = idesc_make(kFmt, 128, kBR, false, false);     // S^T, dP^T
  constexpr uint32_t kIdKV = idesc_make(kFmt, 128, kBwdD, false, true);   // dV, dK
  constexpr uint32_t kIdQ = idesc_make(kFmt, 128, kBR, true, true);       // dQ^T
  extern __shared__ uint8_t bsm_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(bsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
  uint64_t *bar_kv = bars + 0;
  uint64_t *bar_qfull = bars + 1;           // [2]
  uint64_t *bar_qempty = bars + 3;          // [2]
  uint64_t *bar_s = bars + 5;               // S^T and dP^T ready
  uint64_t *bar_pds = bars + 6;             // P^T and dS^T written (S^T, dP^T read)
  uint64_t *bar_dq = bars + 7;              // dV, dK, dQ^T updates done
  uint64_t *bar_dqfree = bars + 8;          // dQ^T read out of TMEM
  uint64_t *bar_final = bars + 9;           // every MMA done
  uint64_t *bar_drain = bars + 10;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int kb = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int key0 = kb * kBC;
  const int g = p.H / p.Hkv;
  const int nqb = (p.N + kBR - 1) / kBR;
  const int qb0 = p.causal ? key0 / kBR : 0;              // first query block that sees a key
  const int n_it = g * (nqb - qb0);                       // (head, query block) iterations

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_qfull[i], 1);
      mbar_init(&bar_qempty[i], 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_pds, 128);
    mbar_init(bar_dq, 1);
    mbar_init(bar_dqfree, 128);
    mbar_init(bar_final, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMMAb) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  if (warp == kWarpTMAb && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const WaitCtl wc{abort_flag, p.status, p.wait_budget};
  // iteration it -> (query head h, query block qb)
  auto it_head = [&](int it) { return hk * g + it / (nqb - qb0); };
  auto it_qb = [&](int it) { return qb0 + it % (nqb - qb0); };

  if (warp == kWarpTMAb) {
    // ------------------------------------------------------------------
    // TMA: K and V of this block once, then Q and dO per iteration
    // ------------------------------------------------------------------
    if (lane == 0) {
      bool ok = true;
      int issued[2] = {0, 0};
      mbar_arrive_expect_tx(bar_kv, 2 * L::kKVBytes);
      for (int c = 0; c < 2; ++c) {
        tma_load_4d(smem + L::kOffK + c * (L::kKVBytes / 2), &tmK, bar_kv, c * 64, hk, key0, b);
        tma_load_4d(smem + L::kOffV + c * (L::kKVBytes / 2), &tmV, bar_kv, c * 64, hk, key0, b);
      }
      for (int it = 0; it < n_it; ++it) {
        const int buf = it & 1;
        if (!mbar_wait(&bar_qempty[buf], ((it >> 1) & 1) ^ 1, wc)) { ok = false; break; }
        const int h = it_head(it), q0 = it_qb(it) * kBR;
        mbar_arrive_expect_tx(&bar_qfull[buf], 2 * L::kQBytes);
        ++issued[buf];
        for (int c = 0; c < 2; ++c) {
          tma_load_4d(smem + L::kOffQ + buf * L::kQBytes + c * (L::kQBytes / 2), &tmQ,
                      &bar_qfull[buf], c * 64, h, q0, b);
          tma_load_4d(smem + L::kOffDO + buf * L::kQBytes + c * (L::kQBytes / 2), &tmDO,
                      &bar_qfull[buf], c * 64, h, q0, b);
        }
      }
      if (!ok) {
        // let every copy this CTA started land before it exits
        mbar_wait_drain(bar_kv, 0);
        for (int buf = 0; buf < 2; ++buf)
          if (issued[buf] > 0) mbar_wait_drain(&bar_qfull[buf], (issued[buf] - 1) & 1);
      }
    }
  } else if (warp == kWarpMMAb) {
    // ------------------------------------------------------------------
    // MMA issuer (one thread)
    // ------------------------------------------------------------------
    if (lane == 0) {
      const uint64_t kK = sdesc_sw128(smem_addr(smem + L::kOffK), 16, 1024);       // K-major A
      const uint64_t kV = sdesc_sw128(smem_addr(smem + L::kOffV), 16, 1024);
      const uint64_t kKt = sdesc_sw128(smem_addr(smem + L::kOffK), L::kKVBytes / 2, 1024);  // MN-major A
      const uint64_t kP = sdesc_sw128(smem_addr(smem + L::kOffP), 16, 1024);
      const uint64_t kDS = sdesc_sw128(smem_addr(smem + L::kOffDS), 16, 1024);
      const uint64_t kDSn = sdesc_sw128(smem_addr(smem + L::kOffDS), 16, 1024);    // MN-major B
      bool ok = mbar_wait(bar_kv, 0, wc);
      tc_fence_after();
      for (int it = 0; ok && it < n_it; ++it) {
        const int buf = it & 1;
        if (!mbar_wait(&bar_qfull[buf], (it >> 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t qa = smem_addr(smem + L::kOffQ + buf * L::kQBytes);
        const uint32_t da = smem_addr(smem + L::kOffDO + buf * L::kQBytes);
        const uint64_t kQ = sdesc_sw128(qa, 16, 1024);                              // K-major B
        const uint64_t kDO = sdesc_sw128(da, 16, 1024);
        const uint64_t kQn = sdesc_sw128(qa, L::kQBytes / 2, 1024);                 // MN-major B
        const uint64_t kDOn = sdesc_sw128(da, L::kQBytes / 2, 1024);
        // S^T = K Q^T and dP^T = V dO^T: K steps of 16 along d (32 bytes in a
        // 128-byte chunk; chunks 16 KB apart in K/V, 8 KB in Q/dO)
#pragma unroll
        for (int s = 0; s < kBwdD / 16; ++s) {
          const uint32_t oa = ((s / 4) * (L::kKVBytes / 2) + (s % 4) * 32) >> 4;
          const uint32_t ob = ((s / 4) * (L::kQBytes / 2) + (s % 4) * 32) >> 4;
          mma_f16_ss(tmem + kColS, kK + oa, kQ + ob, kIdS, s > 0);
          mma_f16_ss(tmem + kColDP, kV + oa, kDO + ob, kIdS, s > 0);
        }
        mma_commit(bar_s);
        // P^T and dS^T in shared memory, and the previous dQ^T read out
        if (!mbar_wait(bar_pds, it & 1, wc)) { ok = false; break; }
        if (it > 0 && !mbar_wait(bar_dqfree, (it - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        // dV += P^T dO and dK += dS^T Q: K steps of 16 query rows (32 bytes
        // of the P^T / dS^T rows; 16 rows = 2 KB of the MN-major dO / Q)
#pragma unroll
        for (int s = 0; s < kBR / 16; ++s) {
          const uint32_t oa = (s * 32) >> 4;
          const uint32_t ob = (s * 16 * 128) >> 4;
          mma_f16_ss(tmem + kColDV, kP + oa, kDOn + ob, kIdKV, it > 0 || s > 0);
          mma_f16_ss(tmem + kColDK, kDS + oa, kQn + ob, kIdKV, it > 0 || s > 0);
        }
        // dQ^T = K^T dS^T: K steps of 16 keys (16 rows = 2 KB of K and of dS^T)
#pragma unroll
        for (int s = 0; s < kBC / 16; ++s) {
          const uint32_t o = (s * 16 * 128) >> 4;
          mma_f16_ss(tmem + kColDQ, kKt + o, kDSn + o, kIdQ, s > 0);
        }
        mma_commit(bar_dq);
        mma_commit(&bar_qempty[buf]);
      }
      mma_commit(bar_final);
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------
    // Softmax warps: thread r = key row of the block (and TMEM lane r)
    // ------------------------------------------------------------------
    const int r = threadIdx.x;                        // 0 .. 127
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int key = key0 + r;
    const uint32_t p_row = smem_addr(smem + L::kOffP) + r * 128;
    const uint32_t ds_row = smem_addr(smem + L::kOffDS) + r * 128;
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it) {
      const int h = it_head(it), q0 = it_qb(it) * kBR;
      const size_t vrow = (static_cast<size_t>(b) * p.H + h) * p.N;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_s, it & 1, wc))) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[64], dp[64];
      tmem_ld64(tmem + lane_base + kColS, sv);
      tmem_ld64(tmem + lane_base + kColDP, dp);
      // the previous block's dV / dK / dQ^T updates have read P^T and dS^T
      // (this thread waited for them when it read dQ^T)
#pragma unroll
      for (int u = 0; u < 8; ++u) {                  // 8 queries per 16-byte unit
        uint32_t pw[4], dw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float pv[2], dv2[2];
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int i = 8 * u + 2 * e + t, q = q0 + i;
            const bool live = key < p.N && q < p.N && (!p.causal || key <= q);
            const float l2 = __ldg(p.lse + vrow + min(q, p.N - 1)) * 1.4426950408889634f;
            const float pp = live ? ex2(__uint_as_float(sv[i]) * p.scale_log2 - l2) : 0.f;
            const float dd = __ldg(p.Dvec + vrow + min(q, p.N - 1));
            pv[t] = pp;
            dv2[t] = pp * (__uint_as_float(dp[i]) - dd);
          }
          pw[e] = (E == Elem::BF16) ? pack_bf16(pv[0], pv[1]) : pack_f16(pv[0], pv[1]);
          dw[e] = (E == Elem::BF16) ? pack_bf16(dv2[0], dv2[1]) : pack_f16(dv2[0], dv2[1]);
        }
        st_shared_v4(p_row + ((u ^ (r & 7)) << 4), pw[0], pw[1], pw[2], pw[3]);
        st_shared_v4(ds_row + ((u ^ (r & 7)) << 4), dw[0], dw[1], dw[2], dw[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_pds);
      // dQ^T: TMEM lane r holds head-dim column r for the 64 queries
      if (!__all_sync(0xffffffffu, mbar_wait(bar_dq, it & 1, wc))) { ok = false; break; }
      tc_fence_after();
      uint32_t dq[64];
      tmem_ld64(tmem + lane_base + kColDQ, dq);
      tc_fence_before();
      mbar_arrive(bar_dqfree);
      float *acc = p.dq_acc + (static_cast<size_t>(b) * p.N * p.H + h) * kBwdD + r;
      for (int i = 0; i < kBR; ++i) {
        const int q = q0 + i;
        if (q < p.N) atomicAdd(acc + static_cast<size_t>(q) * p.H * kBwdD, __uint_as_float(dq[i]));
      }
    }
    // epilogue: dV and dK rows of this key
    if (ok && __all_sync(0xffffffffu, mbar_wait(bar_final, 0, wc))) {
      tc_fence_after();
      const size_t orow = ((static_cast<size_t>(b) * p.N + min(key, p.N - 1)) * p.Hkv + hk) * kBwdD;
      uint16_t *dvo = static_cast<uint16_t *>(p.dv) + orow;
      uint16_t *dko = static_cast<uint16_t *>(p.dk) + orow;
#pragma unroll 1
      for (int c = 0; c < kBwdD / 32; ++c) {
        uint32_t a[32], k2[32];
        tmem_ld32(tmem + lane_base + kColDV + c * 32, a);
        tmem_ld32(tmem + lane_base + kColDK + c * 32, k2);
        if (key < p.N) {
          uint32_t wa[16], wk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a0 = __uint_as_float(a[2 * i]), a1 = __uint_as_float(a[2 * i + 1]);
            const float k0 = __uint_as_float(k2[2 * i]) * p.scale;
            const float k1 = __uint_as_float(k2[2 * i + 1]) * p.scale;
            wa[i] = (E == Elem::BF16) ? pack_bf16(a0, a1) : pack_f16(a0, a1);
            wk[i] = (E == Elem::BF16) ? pack_bf16(k0, k1) : pack_f16(k0, k1);
          }
          uint4 *da = reinterpret_cast<uint4 *>(dvo + c * 32);
          uint4 *dk4 = reinterpret_cast<uint4 *>(dko + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            da[i] = make_uint4(wa[4 * i], wa[4 * i + 1], wa[4 * i + 2], wa[4 * i + 3]);
            dk4[i] = make_uint4(wk[4 * i], wk[4 * i + 1], wk[4 * i + 2], wk[4 * i + 3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMAb) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// D_i = rowsum(dO_i * O_i), one warp per (token, head) row.
template <Elem E>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint16_t *o, const uint16_t *dout,
                                                      float *Dvec, int B, int H, int N) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= B * N * H) return;
  const int h = row % H, t = row / H;                    // t = b * N + n
  const uint2 ov = *reinterpret_cast<const uint2 *>(o + static_cast<size_t>(row) * kBwdD + 4 * lane);
  const uint2 dv = *reinterpret_cast<const uint2 *>(dout + static_cast<size_t>(row) * kBwdD + 4 * lane);
  const uint32_t ow[2] = {ov.x, ov.y}, dw[2] = {dv.x, dv.y};
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float o0, o1, d0, d1;
    if constexpr (E == Elem::BF16) {
      o0 = __uint_as_float(ow[i] << 16); o1 = __uint_as_float(ow[i] & 0xffff0000u);
      d0 = __uint_as_float(dw[i] << 16); d1 = __uint_as_float(dw[i] & 0xffff0000u);
    } else {
      const __half2 oh = *reinterpret_cast<const __half2 *>(&ow[i]);
      const __half2 dh = *reinterpret_cast<const __half2 *>(&dw[i]);
      o0 = __low2float(oh); o1 = __high2float(oh); d0 = __low2float(dh); d1 = __high2float(dh);
    }
    acc = fmaf(o0, d0, fmaf(o1, d1, acc));
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (lane == 0) Dvec[(static_cast<size_t>(t / N) * H + h) * N + t % N] = acc;
}

// dQ = scale * accumulator, rounded to the output type.
template <Elem E>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float *acc, uint16_t *dq, size_t n,
                                                     float scale) {
  const size_t i = (static_cast<size_t>(blockIdx.x) * 256 + threadIdx.x) * 4;
  if (i >= n) return;
  const float4 a = *reinterpret_cast<const float4 *>(acc + i);
  const uint32_t w0 = (E == Elem::BF16) ? pack_bf16(a.x * scale, a.y * scale)
                                        : pack_f16(a.x * scale, a.y * scale);
  const uint32_t w1 = (E == Elem::BF16) ? pack_bf16(a.z * scale, a.w * scale)
                                        : pack_f16(a.z * scale, a.w * scale);
  *reinterpret_cast<uint2 *>(dq + i) = make_uint2(w0, w1);
}

template <Elem E>
attn_status_t launch_bwd(const void *q, const void *k, const void *v, const void *o,
                         const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                         int H, int Hkv, int N, float scale, int causal, DeviceState *ds,
                         cudaStream_t s) {
  const size_t nq = static_cast<size_t>(B) * N * H * kBwdD;
  const size_t rows = static_cast<size_t>(B) * H * N;
  attn_status_t st = ensure_bwd_workspace(ds, (nq + rows) * sizeof(float));
  if (st != ATTN_OK) return st;
  float *acc = ds->bwd_ws;
  float *Dvec = ds->bwd_ws + nq;
  if (cudaMemsetAsync(acc, 0, nq * sizeof(float), s) != cudaSuccess) return ATTN_ERR_CUDA;
  bwd_pre_kernel<E><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(
      static_cast<const uint16_t *>(o), static_cast<const uint16_t *>(dout), Dvec, B, H, N);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  const CUtensorMapDataType dt =
      E == Elem::BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mq, mk, mv, mdo;
  auto map = [&](CUtensorMap *m, const void *ptr, int heads, int rows_box) {
    const cuuint64_t dims[4] = {(cuuint64_t)kBwdD, (cuuint64_t)heads, (cuuint64_t)N,
                                (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)kBwdD * 2, (cuuint64_t)heads * kBwdD * 2,
                                   (cuuint64_t)N * heads * kBwdD * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)rows_box, 1};
    return encode_tiled(m, dt, 4, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  };
  if ((st = map(&mq, q, H, kBR)) != ATTN_OK || (st = map(&mdo, dout, H, kBR)) != ATTN_OK ||
      (st = map(&mk, k, Hkv, kBC)) != ATTN_OK || (st = map(&mv, v, Hkv, kBC)) != ATTN_OK)
    return st;
  BwdParams p{};
  p.lse = lse; p.Dvec = Dvec; p.dq_acc = acc; p.dk = dk; p.dv = dv;
  p.B = B; p.H = H; p.Hkv = Hkv; p.N = N;
  p.scale = scale; p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = causal ? 1 : 0;
  p.wait_budget = wait_budget();
  p.status = ds->status;
  static std::once_flag once[kMaxDevices];
  static cudaError_t err[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::call_once(once[dev], [dev] {
    err[dev] = cudaFuncSetAttribute(bwd_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    BwdSmem::kBytes);
  });
  if (err[dev] != cudaSuccess) return ATTN_ERR_LAUNCH;
  bwd_kernel<E><<<dim3((N + kBC - 1) / kBC, Hkv, B), kBwdThreads, BwdSmem::kBytes, s>>>(
      mq, mk, mv, mdo, p);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  bwd_dq_kernel<E><<<static_cast<unsigned>((nq / 4 + 255) / 256), 256, 0, s>>>(
      acc, static_cast<uint16_t *>(dq), nq, scale);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" attn_status_t attn_bwd(const void *q, const void *k, const void *v, const void *o,
                                  const void *dout, const float *lse, void *dq, void *dk,
                                  void *dv, int B, int H, int H_kv, int N, int d, float scale,
                                  int causal, attn_dtype_t dtype, void *stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || H < 1 || H_kv < 1 || H % H_kv != 0 || !std::isfinite(scale))
    return ATTN_ERR_INVALID_ARG;
  if (d != kBwdD) return ATTN_ERR_UNSUPPORTED;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return ATTN_ERR_MISALIGNED;
  if (static_cast<long long>(B) * N * H * d > (1LL << 36)) return ATTN_ERR_TOO_LARGE;
  DeviceState *ds = nullptr;
  attn_status_t st = device_state(&ds);
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return dtype == ATTN_BF16
             ? launch_bwd<Elem::BF16>(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N, scale,
                                      causal, ds, s)
             : launch_bwd<Elem::F16>(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N, scale,
                                     causal, ds, s);
}
