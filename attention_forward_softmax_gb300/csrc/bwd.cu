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
//    key row) have turned them into P^T (written back to TMEM over the dP^T
//    columns they have read) and dS^T (shared memory) -- dV += P^T dO (P^T
//    from TMEM, as P in the forward's P V), dK += dS^T Q (dO and Q read
//    MN-major, as V in the forward), and dQ^T = K^T dS^T (K read MN-major as
//    the A operand);
//  * two TMEM buffers hold S^T | dP^T of consecutive blocks, two
//    shared-memory slots their dS^T, and a three-deep ring Q and dO: the MMA
//    warp computes S^T of block i+2 while the softmax warps work on block
//    i+1 and the tensor pipe finishes the products of block i, and the copy
//    of block i+2 was started a block earlier.  dQ^T of block i is written
//    over the S^T columns of its buffer, once the softmax warps have read
//    them;
//  * four dQ warps read dQ^T out of TMEM (one thread per head-dim column),
//    stage it as an fp32 [64 x 128] tile and add it to an fp32 accumulator in
//    global memory with one bulk tensor reduce; a last pass scales it and
//    rounds it to the output type;
//  * TMEM: buffer j = columns [128 j, 128 j + 128): S^T (then dQ^T) in the
//    first 64, dP^T (then P^T, two 16-bit values per column) in the next 64;
//    dV [256,384), dK [384,512);
//  * every mbarrier wait is bounded; on expiry the status word gets
//    ATTN_ERR_TIMEOUT, every role leaves its loop at the same named-barrier
//    step, and the CTA drains its copies and MMAs and returns.
#include <climits>
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
constexpr int kBwdThreads = 320;            // 4 softmax warps, MMA, TMA, 4 dQ warps
constexpr int kWarpMMAb = 4, kWarpTMAb = 5, kWarpDQ0 = 6;
constexpr uint32_t kBarSoftmax = 1, kBarDQ = 2;   // named barriers (128 threads each)

struct BwdParams {
  const float *lse;                         // [B, H, N] natural log
  const float *Dvec;                        // [B, H, N] rowsum(dO * O)
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
  static constexpr int kDQBytes = kBR * kBwdD * 4;        // 32 KB: fp32 [64][128]
  static constexpr int kNQ = 3;                           // Q / dO ring depth
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKVBytes;
  static constexpr int kOffQ = kOffV + kKVBytes;          // [kNQ buffers]
  static constexpr int kOffDO = kOffQ + kNQ * kQBytes;    // [kNQ buffers]
  static constexpr int kOffDS = kOffDO + kNQ * kQBytes;   // [2 slots]
  static constexpr int kOffDQ = kOffDS + 2 * kPBytes;
  static constexpr int kOffStage = kOffDQ + kDQBytes;     // [2 slots] of -lse*log2e | -D
  static constexpr int kOffBar = kOffStage + 2 * 128 * 4;
  static constexpr int kNumBars = 20;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 64 + 1024;     // + alignment slack
  static_assert(kBytes <= 227 * 1024, "backward tile set exceeds the shared memory of a CTA");
};

constexpr uint32_t kColBuf = 128, kColDP = 64, kColDV = 256, kColDK = 384;

// P^T and dS^T for 32 queries (columns [32 half, 32 half + 32)) of this
// thread's key row: P^T packed in pairs into pw, dS^T written as four 16-byte
// units of its swizzled shared-memory row.  `sl` holds -lse*log2e for the 64
// queries, then -D.  Masked: query column i is live iff i >= thr.
template <Elem E, bool Masked>
__device__ __forceinline__ void bwd_softmax_half(const uint32_t (&sv)[32], const uint32_t (&dp)[32],
                                                 const float *sl, float c, int thr, int half,
                                                 uint32_t ds_row, int r, uint32_t (&pw)[16]) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i0 = half * 32 + u * 8;
    const float4 l0 = *reinterpret_cast<const float4 *>(sl + i0);
    const float4 l1 = *reinterpret_cast<const float4 *>(sl + i0 + 4);
    const float4 d0 = *reinterpret_cast<const float4 *>(sl + 64 + i0);
    const float4 d1 = *reinterpret_cast<const float4 *>(sl + 64 + i0 + 4);
    const float nl[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
    const float nd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
    uint32_t dw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = u * 8 + 2 * e;              // index within this half
      float x0, x1, t0, t1;
      ffma2(x0, x1, __uint_as_float(sv[j]), __uint_as_float(sv[j + 1]), c, c, nl[2 * e],
            nl[2 * e + 1]);
      float p0 = ex2(x0), p1 = ex2(x1);
      if (Masked) {
        if (i0 + 2 * e < thr) p0 = 0.f;
        if (i0 + 2 * e + 1 < thr) p1 = 0.f;
      }
      fadd2(t0, t1, __uint_as_float(dp[j]), __uint_as_float(dp[j + 1]), nd[2 * e], nd[2 * e + 1]);
      const float g0 = p0 * t0, g1 = p1 * t1;
      pw[u * 4 + e] = (E == Elem::BF16) ? pack_bf16(p0, p1) : pack_f16(p0, p1);
      dw[e] = (E == Elem::BF16) ? pack_bf16(g0, g1) : pack_f16(g0, g1);
    }
    const uint32_t off = (static_cast<uint32_t>(half * 4 + u) ^ static_cast<uint32_t>(r & 7)) << 4;
    st_shared_v4(ds_row + off, dw[0], dw[1], dw[2], dw[3]);
  }
}

// One 128-column TMEM accumulator row (this thread's key) times `mul`,
// rounded and stored as a row of d 16-bit values.
template <Elem E>
__device__ __forceinline__ void bwd_store_row(uint32_t taddr, uint16_t *dst, float mul, bool live) {
#pragma unroll 1
  for (int c = 0; c < kBwdD / 32; ++c) {
    uint32_t a[32];
    tmem_ld32(taddr + c * 32, a);
    if (live) {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float a0 = __uint_as_float(a[2 * i]) * mul, a1 = __uint_as_float(a[2 * i + 1]) * mul;
        w[i] = (E == Elem::BF16) ? pack_bf16(a0, a1) : pack_f16(a0, a1);
      }
      uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
  }
}

template <Elem E>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ BwdParams p) {
  using L = BwdSmem;
  constexpr uint32_t kFmt = (E == Elem::BF16) ? 1u : 0u;
  constexpr uint32_t kIdS = idesc_make(kFmt, 128, kBR, false, false);     // S^T, dP^T
  constexpr uint32_t kIdKV = idesc_make(kFmt, 128, kBwdD, false, true);   // dV, dK
  constexpr uint32_t kIdQ = idesc_make(kFmt, 128, kBR, true, true);       // dQ^T
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ uint8_t bsm_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(bsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
  uint64_t *bar_kv = bars + 0;
  constexpr int NQ = L::kNQ;
  uint64_t *bar_qfull = bars + 1;           // [NQ] Q, dO of a block landed
  uint64_t *bar_qempty = bars + 1 + NQ;     // [NQ] Q, dO buffer read by every MMA
  uint64_t *bar_sfull = bars + 1 + 2 * NQ;  // [2] S^T, dP^T in the TMEM buffer
  uint64_t *bar_pds = bar_sfull + 2;        // [2] P^T, dS^T written (S^T, dP^T read)
  uint64_t *bar_dqfull = bar_pds + 2;       // [2] dV, dK, dQ^T updates of a block done
  uint64_t *bar_dqfree = bar_dqfull + 2;    // [2] dQ^T read out of the TMEM buffer
  uint64_t *bar_final = bar_dqfree + 2;     // every MMA done
  uint64_t *bar_drain = bar_final + 1;
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
    for (int i = 0; i < NQ; ++i) {
      mbar_init(&bar_qfull[i], 1);
      mbar_init(&bar_qempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_sfull[i], 1);
      mbar_init(&bar_pds[i], 128);
      mbar_init(&bar_dqfull[i], 1);
      mbar_init(&bar_dqfree[i], 128);
    }
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
    tma_prefetch_desc(&tmDQ);
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
      int issued[NQ] = {};
      mbar_arrive_expect_tx(bar_kv, 2 * L::kKVBytes);
      for (int c = 0; c < 2; ++c) {
        tma_load_4d(smem + L::kOffK + c * (L::kKVBytes / 2), &tmK, bar_kv, c * 64, hk, key0, b);
        tma_load_4d(smem + L::kOffV + c * (L::kKVBytes / 2), &tmV, bar_kv, c * 64, hk, key0, b);
      }
      for (int it = 0; it < n_it; ++it) {
        const int buf = it % NQ;
        if (!mbar_wait(&bar_qempty[buf], ((it / NQ) & 1) ^ 1, wc)) { ok = false; break; }
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
        for (int buf = 0; buf < NQ; ++buf)
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
      // S^T = K Q^T and dP^T = V dO^T of block j into TMEM buffer j & 1:
      // K steps of 16 along d (32 bytes in a 128-byte chunk; chunks 16 KB
      // apart in K/V, 8 KB in Q/dO)
      auto issue_s = [&](int j) {
        const int buf = j & 1, qbuf = j % NQ;
        const uint64_t kQ = sdesc_sw128(smem_addr(smem + L::kOffQ + qbuf * L::kQBytes), 16, 1024);
        const uint64_t kDO = sdesc_sw128(smem_addr(smem + L::kOffDO + qbuf * L::kQBytes), 16, 1024);
        const uint32_t ts = tmem + buf * kColBuf;
#pragma unroll
        for (int s = 0; s < kBwdD / 16; ++s) {
          const uint32_t oa = ((s / 4) * (L::kKVBytes / 2) + (s % 4) * 32) >> 4;
          const uint32_t ob = ((s / 4) * (L::kQBytes / 2) + (s % 4) * 32) >> 4;
          mma_f16_ss(ts, kK + oa, kQ + ob, kIdS, s > 0);
          mma_f16_ss(ts + kColDP, kV + oa, kDO + ob, kIdS, s > 0);
        }
        mma_commit(&bar_sfull[buf]);
      };
      bool ok = mbar_wait(bar_kv, 0, wc);
      tc_fence_after();
      for (int j = 0; ok && j < 2 && j < n_it; ++j) {
        if (!mbar_wait(&bar_qfull[j % NQ], 0, wc)) { ok = false; break; }
        tc_fence_after();
        issue_s(j);
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const int buf = it & 1, qbuf = it % NQ;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(&bar_pds[buf], ph, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tPt = tmem + buf * kColBuf + kColDP;                          // P^T, TMEM
        const uint64_t kDS = sdesc_sw128(smem_addr(smem + L::kOffDS + buf * L::kPBytes), 16, 1024);
        const uint64_t kQn =
            sdesc_sw128(smem_addr(smem + L::kOffQ + qbuf * L::kQBytes), L::kQBytes / 2, 1024);
        const uint64_t kDOn =
            sdesc_sw128(smem_addr(smem + L::kOffDO + qbuf * L::kQBytes), L::kQBytes / 2, 1024);
        // dV += P^T dO and dK += dS^T Q: K steps of 16 query rows (8 TMEM
        // columns of P^T; 32 bytes of the dS^T rows; 16 rows = 2 KB of the
        // MN-major dO / Q)
#pragma unroll
        for (int s = 0; s < kBR / 16; ++s) {
          const uint32_t oa = (s * 32) >> 4;
          const uint32_t ob = (s * 16 * 128) >> 4;
          mma_f16_ts(tmem + kColDV, tPt + s * 8, kDOn + ob, kIdKV, it > 0 || s > 0);
          mma_f16_ss(tmem + kColDK, kDS + oa, kQn + ob, kIdKV, it > 0 || s > 0);
        }
        // dQ^T = K^T dS^T over the S^T columns of this buffer: K steps of 16
        // keys (16 rows = 2 KB of K and of dS^T, the latter read MN-major)
#pragma unroll
        for (int s = 0; s < kBC / 16; ++s) {
          const uint32_t o = (s * 16 * 128) >> 4;
          mma_f16_ss(tmem + buf * kColBuf, kKt + o, kDS + o, kIdQ, s > 0);
        }
        mma_commit(&bar_dqfull[buf]);
        mma_commit(&bar_qempty[qbuf]);
        if (it + 2 < n_it) {
          // block it + 2 reuses this TMEM buffer
          if (!mbar_wait(&bar_qfull[(it + 2) % NQ], ((it + 2) / NQ) & 1, wc)) { ok = false; break; }
          if (!mbar_wait(&bar_dqfree[buf], ph, wc)) { ok = false; break; }
          tc_fence_after();
          issue_s(it + 2);
        }
      }
      mma_commit(bar_final);
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------------
    // Softmax warps: thread r = key row of the block (and TMEM lane r)
    // ------------------------------------------------------------------
    const int r = threadIdx.x;                        // 0 .. 127
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int key = key0 + r;
    float *stage = reinterpret_cast<float *>(smem + L::kOffStage);
    // threads 0-63 stage -lse*log2e of query q0 + r (-inf past the end, so
    // P = 0 there), threads 64-127 stage -D of query q0 + r - 64
    auto stage_val = [&](int j) -> float {
      const int h = it_head(j), q = it_qb(j) * kBR + (r & 63);
      const size_t row = (static_cast<size_t>(b) * p.H + h) * p.N;
      if (q >= p.N) return r < 64 ? -INFINITY : 0.f;
      return r < 64 ? -__ldg(p.lse + row + q) * kLog2e : -__ldg(p.Dvec + row + q);
    };
    float nxt = stage_val(0);
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it) {
      const int buf = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      const int q0 = it_qb(it) * kBR;
      stage[buf * 128 + r] = nxt;
      if (it + 1 < n_it) nxt = stage_val(it + 1);
      // the P^T / dS^T slot is free once the MMAs of block it - 2 are done
      bool w = true;
      if (it >= 2) w = mbar_wait(&bar_dqfull[buf], ph ^ 1, wc);
      w = w && mbar_wait(&bar_sfull[buf], ph, wc);
      // (the barrier also publishes the staged values)
      if (!named_bar_and(kBarSoftmax, 128, w)) { ok = false; break; }
      tc_fence_after();
      const float *sl = stage + buf * 128;
      const uint32_t tS = tmem + lane_base + buf * kColBuf;
      const uint32_t ds_row = smem_addr(smem + L::kOffDS + buf * L::kPBytes) + r * 128;
      // masking only where a block has keys past the end or above the
      // causal diagonal
      const bool masked = (p.causal && q0 < key0 + kBC - 1) || key0 + kBC > p.N;
      const int thr = key < p.N ? (p.causal ? key - q0 : INT_MIN) : INT_MAX;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t sv[32], dp[32], pw[16];
        tmem_ld32x2(tS + half * 32, tS + kColDP + half * 32, sv, dp);
        if (masked)
          bwd_softmax_half<E, true>(sv, dp, sl, p.scale_log2, thr, half, ds_row, r, pw);
        else
          bwd_softmax_half<E, false>(sv, dp, sl, p.scale_log2, thr, half, ds_row, r, pw);
        // P^T over dP^T columns this thread has already read (half 0's)
        tmem_st16_nowait(tS + kColDP + half * 16, pw);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_pds[buf]);
    }
    // epilogue: the dV row of this key
    if (ok && __all_sync(0xffffffffu, mbar_wait(bar_final, 0, wc))) {
      tc_fence_after();
      const size_t orow = ((static_cast<size_t>(b) * p.N + min(key, p.N - 1)) * p.Hkv + hk) * kBwdD;
      bwd_store_row<E>(tmem + lane_base + kColDV, static_cast<uint16_t *>(p.dv) + orow, 1.f,
                       key < p.N);
    }
  } else {
    // ------------------------------------------------------------------
    // dQ warps: thread = head-dim column (TMEM lane) of dQ^T
    // ------------------------------------------------------------------
    const int sub = warp & 3;                         // TMEM lane quarter of this warp
    const int col = sub * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(sub * 32) << 16;
    const bool leader = threadIdx.x == kWarpDQ0 * 32;
    float *tile = reinterpret_cast<float *>(smem + L::kOffDQ);
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it) {
      const int buf = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      // dQ^T out of TMEM first, so the MMA warp can reuse the buffer while
      // this block's reduce waits for the previous one
      const bool w = __all_sync(0xffffffffu, mbar_wait(&bar_dqfull[buf], ph, wc));
      uint32_t v0[32], v1[32];
      if (w) {
        tc_fence_after();
        const uint32_t tq = tmem + lane_base + buf * kColBuf;
        tmem_ld32x2(tq, tq + 32, v0, v1);
        tc_fence_before();
        mbar_arrive(&bar_dqfree[buf]);
      }
      // the previous block's reduce has read the staging tile
      if (leader) bulk_wait_group_read<0>();
      if (!named_bar_and(kBarDQ, 128, w)) { ok = false; break; }
#pragma unroll
      for (int i = 0; i < 32; ++i) tile[i * kBwdD + col] = __uint_as_float(v0[i]);
#pragma unroll
      for (int i = 0; i < 32; ++i) tile[(32 + i) * kBwdD + col] = __uint_as_float(v1[i]);
      fence_proxy_async_smem();
      named_bar_sync(kBarDQ, 128);
      if (leader) {
        tma_reduce_add_4d(&tmDQ, tile, 0, it_head(it), it_qb(it) * kBR, b);
        bulk_commit_group();
      }
    }
    if (leader) bulk_wait_group<0>();
    // epilogue: the dK row of key key0 + col
    const int key = key0 + col;
    if (ok && __all_sync(0xffffffffu, mbar_wait(bar_final, 0, wc))) {
      tc_fence_after();
      const size_t orow = ((static_cast<size_t>(b) * p.N + min(key, p.N - 1)) * p.Hkv + hk) * kBwdD;
      bwd_store_row<E>(tmem + lane_base + kColDK, static_cast<uint16_t *>(p.dk) + orow, p.scale,
                       key < p.N);
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
  // the fp32 dQ accumulator, [B, N, H, d], one unswizzled [64 x 128] box
  CUtensorMap mdq;
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kBwdD, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)kBwdD * 4, (cuuint64_t)H * kBwdD * 4,
                                   (cuuint64_t)N * H * kBwdD * 4};
    const cuuint32_t box[4] = {(cuuint32_t)kBwdD, 1, (cuuint32_t)kBR, 1};
    if ((st = encode_tiled(&mdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, acc, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_NONE)) != ATTN_OK)
      return st;
  }
  BwdParams p{};
  p.lse = lse; p.Dvec = Dvec; p.dk = dk; p.dv = dv;
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
      mq, mk, mv, mdo, mdq, p);
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
