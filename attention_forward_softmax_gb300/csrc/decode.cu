// decode.cu -- attention of a few new queries per sequence against a paged
// K/V cache, split over key ranges, and the merge of the partial results
// (the inference variants the pages point to: "Paged Attention" among the
// additions of the HippoAttention case study, streamhpc.com, "Our
// approach"; "optimizing for LLM inference", FlashAttention-3 summary,
// arxivlens, Limitations).
//
// What it computes is exact attention (the "Fused attention kernel" concept
// card, Overview): for each query row, softmax(scale * q K^T) V and the
// natural-log lse over the allowed keys of its sequence.  The keys of
// sequence b are its first seqlens_k[b] cache positions; position t lives in
// row t % page_size of page block_table[b][t / page_size].  The Nq queries
// are the last Nq positions (causal: query i sees keys j <= L - Nq + i).
// Query head h uses K/V head h / (H / H_kv).
//
// Design.  Decoding is bound by HBM: each key brings 4 d bytes of K and V
// and meets only the R = (H / H_kv) * Nq query rows of its K/V head.  So one
// CTA takes one (sequence, K/V head, key range) and streams that range once:
//  * 64-key tiles of K and V arrive through the page table, two stages per
//    CTA and three CTAs per SM, so the next tile is in flight while this one
//    is used (measured: more CTAs per SM beat deeper stages in fewer CTAs).
//    When a page splits into pieces of 16, 32 or 64 rows, one thread copies
//    each piece with a tensor copy (a box of those rows and 64 columns of
//    the cache seen as a (d, H_kv, pages * page_size) tensor, 128-byte
//    swizzle) completing on the stage's mbarrier; other page sizes gather
//    rows with 16-byte cp.async copies into XOR-swizzled tiles.  The
//    mbarrier waits are bounded: on expiry the CTA records ATTN_ERR_TIMEOUT,
//    lets its copies land and returns;
//  * the key range of a sequence is cut into chunks of equal size, one per
//    CTA, so long and short sequences spread evenly over the SMs;
//  * the R <= 16 query rows are one 16-row MMA tile; each of the four warps
//    takes 16 keys of a tile and runs the running-softmax loop on them with
//    warp-level bf16/fp16 MMAs (m16n8k16: S = Q K^T, then O += P V with P
//    taken from the score registers).  The contractions are tiny -- 16 rows
//    -- so the tensor pipe is nowhere near the limit; the bytes are;
//  * the four warps' (max, sum, O) are merged through shared memory; with one
//    split the CTA writes O and lse, otherwise fp32 partials that
//    merge_kernel combines: lse = log sum_s exp(lse_s), O = sum_s
//    exp(lse_s - lse) O_s.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kDecThreads = 128;
constexpr int kTileKeys = 64;      // keys per tile (16 per warp)
constexpr int kStages = 2;         // tiles in flight or in use (3 CTAs per SM)
constexpr int kRows = 16;          // query rows per CTA (one MMA tile)

struct DecodeArgs {
  const void *q;                   // [B, Nq, H, d]
  const void *k, *v;               // [num_pages, page_size, H_kv, d]
  const int *block_table;          // [B, max_pages]
  const int *seqlens_k;            // [B]
  void *o;                         // [B, Nq, H, d]
  float *lse;                      // [B, H, Nq] or null
  float *ws_o;                     // [splits, B, H, Nq, d] fp32 partials (splits > 1)
  float *ws_lse;                   // [splits, B, H, Nq]
  int B, Nq, H, Hkv, page_size, max_pages, num_pages;
  int splits;                      // CTAs per (sequence, K/V head): ceil(max_seqlen_k / chunk)
  int chunk;                       // keys per CTA (a multiple of kTileKeys)
  int box_rows;                    // tensor-copy path: cache rows per copy (16, 32 or 64)
  float scale_log2;
  int causal;
  int *status;                     // device status word
  long long budget;                // clock64 cycles per pipeline wait
};

template <int D>
struct DecSmem {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kTileBytes = kTileKeys * kRowBytes;     // one K or V tile
  static constexpr int kOffQ = 0;                              // 16 rows
  static constexpr int kOffKV = kRows * kRowBytes;             // [stage][K, V], 1024-aligned
  static constexpr int kBytes = kOffKV + kStages * 2 * kTileBytes + 1024;   // + alignment slack
  // after the key loop the K/V area holds the warps' partial results
  static_assert(4 * kRows * (D + 2) * 4 <= kStages * 2 * kTileBytes, "merge area too small");
};

// 16-byte chunk c of row r of a swizzled tile (rows of D 16-bit values):
// chunk c is stored at c ^ (r mod 8), so 8 rows read at one chunk hit 8
// different bank groups.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return r * (D * 2) + ((c ^ (r & 7)) << 4);
}

// The same for a K or V tile: row-gathered tiles use swz; tiles written by
// tensor copies hold D / 64 column blocks of 64 rows x 128 bytes, each with
// the copy's 128-byte swizzle (16-byte unit u of row r at u ^ (r mod 8)).
template <int D, bool kTma>
__device__ __forceinline__ uint32_t kv_swz(int r, int c) {
  if constexpr (kTma)
    return (c >> 3) * (kTileKeys * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
  else
    return swz<D>(r, c);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D(16x8, f32) += A(16x16) * B(16x8), 16-bit operands
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (BF16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int D, bool BF16, bool kTma>
__global__ void __launch_bounds__(kDecThreads)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeArgs a) {
  using L = DecSmem<D>;
  constexpr int kChunks = D / 8;           // 16-byte chunks per row
  constexpr int kNT = D / 8;               // 8-column output tiles
  extern __shared__ uint8_t dsm_raw[];
  uint8_t *dsm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(dsm);
  __shared__ uint64_t full[kStages];       // tensor-copy path: a stage's copies landed
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int g = a.H / a.Hkv;               // query heads per K/V head
  const int R = g * a.Nq;                  // query rows of this K/V head (<= 16)
  const int Lk = __ldg(a.seqlens_k + b);
  // key range of this CTA: chunk `split` of the sequence (whole tiles)
  const int k0 = split * a.chunk;
  if (k0 >= Lk && split > 0) return;       // past the end: the merge does not read it
  const int k1 = min(Lk, k0 + a.chunk);
  const int t0 = k0 / kTileKeys, t1 = (k1 + kTileKeys - 1) / kTileKeys;
  const size_t row_stride = static_cast<size_t>(a.Hkv) * D;   // elements between cache rows
  const uint16_t *kc = static_cast<const uint16_t *>(a.k);
  const uint16_t *vc = static_cast<const uint16_t *>(a.v);
  if constexpr (kTma) {
    if (threadIdx.x == 0) {
      for (int i = 0; i < kStages; ++i) mbar_init(&full[i], 1);
      abort_flag = 0;
      fence_mbar_init();
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    __syncthreads();
  }
  const WaitCtl wc{&abort_flag, a.status, a.budget};

  // query rows r = qi * g + gh (query qi, head hk * g + gh) -> shared memory
  {
    const uint16_t *qg = static_cast<const uint16_t *>(a.q);
    for (int id = threadIdx.x; id < kRows * kChunks; id += kDecThreads) {
      const int r = id / kChunks, c = id % kChunks;
      const int qi = r / g, gh = r % g;
      const uint16_t *src = qg + ((static_cast<size_t>(b) * a.Nq + (r < R ? qi : 0)) * a.H +
                                  hk * g + (r < R ? gh : 0)) * D + c * 8;
      cp_async16(sbase + L::kOffQ + swz<D>(r, c), src, r < R ? 16 : 0);
    }
  }
  // one tile of K and V by tensor copies (one thread): a copy per box_rows
  // cache rows (they lie in one page) and 64 columns; copies that would
  // start at or past the end of the range are left out
  auto issue_tile = [&](int tile, int stage) {
    uint8_t *kdst = dsm + L::kOffKV + stage * 2 * L::kTileBytes;
    uint8_t *vdst = kdst + L::kTileBytes;
    const int br = a.box_rows;
    int pieces = 0;
    for (int pc = 0; pc < kTileKeys / br; ++pc)
      if (tile * kTileKeys + pc * br < k1) ++pieces;
    mbar_arrive_expect_tx(&full[stage], pieces * br * D * 2 * 2);
    for (int pc = 0; pc < pieces; ++pc) {
      const int t = tile * kTileKeys + pc * br;
      const int page = __ldg(a.block_table + static_cast<size_t>(b) * a.max_pages + t / a.page_size);
      const int row = page * a.page_size + t % a.page_size;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int off = c * (kTileKeys * 128) + pc * br * 128;
        tma_load_3d(kdst + off, &tmK, &full[stage], c * 64, hk, row);
        tma_load_3d(vdst + off, &tmV, &full[stage], c * 64, hk, row);
      }
    }
  };
  // gather one tile of K and V through the page table
  auto load_tile = [&](int tile, int stage) {
    const uint32_t kdst = sbase + L::kOffKV + stage * 2 * L::kTileBytes;
    const uint32_t vdst = kdst + L::kTileBytes;
    for (int id = threadIdx.x; id < kTileKeys * kChunks; id += kDecThreads) {
      const int r = id / kChunks, c = id % kChunks;
      const int t = tile * kTileKeys + r;
      const bool ok = t < k1;
      const int page = ok ? __ldg(a.block_table + static_cast<size_t>(b) * a.max_pages +
                                  t / a.page_size)
                          : 0;
      const size_t row = ok ? static_cast<size_t>(page) * a.page_size + t % a.page_size : 0;
      const size_t off = row * row_stride + static_cast<size_t>(hk) * D + c * 8;
      cp_async16(kdst + swz<D>(r, c), kc + off, ok ? 16 : 0);
      cp_async16(vdst + swz<D>(r, c), vc + off, ok ? 16 : 0);
    }
  };

  // per-warp running state for the 16 rows: lane holds rows ra = lane/4 and
  // rb = ra + 8 of every accumulator tile
  const int ra = lane >> 2, rb = ra + 8, tq = lane & 3;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  float o[kNT][4];
#pragma unroll
  for (int n = 0; n < kNT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  // last allowed key of each row (causal: queries are the last Nq positions)
  const int lim_a = a.causal ? Lk - a.Nq + ra / g : Lk - 1;
  const int lim_b = a.causal ? Lk - a.Nq + rb / g : Lk - 1;

  // prologue: the first kStages - 1 tiles (row gathers: one commit group per
  // tile, empty groups included, so the group count per tile stays fixed)
  if constexpr (kTma) {
    if (threadIdx.x == 0)
      for (int i = 0; i < kStages - 1; ++i)
        if (t0 + i < t1) issue_tile(t0 + i, i);
    cp_async_commit();                     // the Q rows
  } else {
#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) {
      if (t0 + i < t1) load_tile(t0 + i, i);
      cp_async_commit();
    }
  }
  uint32_t qf[D / 16][4];                  // Q fragments, loaded once
  bool ok = true;
  int tile = t0;
  for (; tile < t1; ++tile) {
    const int stage = (tile - t0) % kStages;
    const int nxt = tile + kStages - 1, nstage = (tile - t0 + kStages - 1) % kStages;
    if constexpr (kTma) {
      // refill the stage read one iteration ago (freed by its closing
      // barrier; its generic reads ordered before the copy)
      if (threadIdx.x == 0 && nxt < t1) {
        fence_proxy_async_smem();
        issue_tile(nxt, nstage);
      }
      if (tile == t0) cp_async_wait<0>();
      const bool got = mbar_wait(&full[stage], ((tile - t0) / kStages) & 1, wc);
      if (!__syncthreads_and(got)) { ok = false; break; }
    } else {
      // refill the stage read one iteration ago (freed by its closing barrier)
      if (nxt < t1) load_tile(nxt, nstage);
      cp_async_commit();
      cp_async_wait<kStages - 1>();
      __syncthreads();
    }
    const uint32_t kt = sbase + L::kOffKV + stage * 2 * L::kTileBytes;
    const uint32_t vt = kt + L::kTileBytes;
    if (kTma && tile * kTileKeys + kTileKeys > k1) {
      // keys at or past the end of the range: their V rows may hold another
      // tile's values or rows of the page past the sequence; zero them (P is
      // 0 there, and 0 * V must be 0)
      const int r0 = max(0, k1 - tile * kTileKeys);
      for (int id = threadIdx.x; id < (kTileKeys - r0) * kChunks; id += kDecThreads)
        st_shared_v4(vt + kv_swz<D, kTma>(r0 + id / kChunks, id % kChunks), 0u, 0u, 0u, 0u);
      fence_proxy_async_smem();            // before a later copy into this stage
      __syncthreads();
    }
    if (tile == t0) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        ldsm_x4(sbase + L::kOffQ + swz<D>(lane & 15, 2 * ks + (lane >> 4)), qf[ks]);
    }
    const int kw = warp * 16;              // this warp's keys within the tile
    // S = Q K^T for 16 keys: two 8-key tiles (one ldmatrix per k step)
    float s[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t kb[4];
      const int key = kw + (lane & 7) + ((lane >> 4) << 3);
      ldsm_x4(kt + kv_swz<D, kTma>(key, 2 * ks + ((lane >> 3) & 1)), kb);
      mma16816<BF16>(s[0], qf[ks], kb[0], kb[1]);
      mma16816<BF16>(s[1], qf[ks], kb[2], kb[3]);
    }
    // mask, then the running softmax in log2 units
    const int kbase = tile * kTileKeys + kw;
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = kbase + n * 8 + 2 * tq + e;
        s[n][e] = (key <= lim_a && key < k1) ? s[n][e] * a.scale_log2 : -INFINITY;
        s[n][2 + e] = (key <= lim_b && key < k1) ? s[n][2 + e] * a.scale_log2 : -INFINITY;
        mx_a = fmaxf(mx_a, s[n][e]);
        mx_b = fmaxf(mx_b, s[n][2 + e]);
      }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, m));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, m));
    }
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float al_a = mn_a == -INFINITY ? 1.f : ex2(m_a - mn_a);
    const float al_b = mn_b == -INFINITY ? 1.f : ex2(m_b - mn_b);
    const float mu_a = mn_a == -INFINITY ? 0.f : mn_a, mu_b = mn_b == -INFINITY ? 0.f : mn_b;
    m_a = mn_a;
    m_b = mn_b;
    float ps_a = 0.f, ps_b = 0.f;
    uint32_t pf[1][4];                     // P as the A fragment of one 16-key step
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      const float p0 = ex2(s[n][0] - mu_a), p1 = ex2(s[n][1] - mu_a);
      const float p2 = ex2(s[n][2] - mu_b), p3 = ex2(s[n][3] - mu_b);
      ps_a += p0 + p1;
      ps_b += p2 + p3;
      const uint32_t pa = BF16 ? pack_bf16(p0, p1) : pack_f16(p0, p1);
      const uint32_t pb = BF16 ? pack_bf16(p2, p3) : pack_f16(p2, p3);
      pf[n >> 1][(n & 1) * 2 + 0] = pa;   // rows ra: keys 2t.. (+8 for the odd tile)
      pf[n >> 1][(n & 1) * 2 + 1] = pb;   // rows rb
    }
    l_a = l_a * al_a + ps_a;
    l_b = l_b * al_b + ps_b;
#pragma unroll
    for (int n = 0; n < kNT; ++n) {
      o[n][0] *= al_a;
      o[n][1] *= al_a;
      o[n][2] *= al_b;
      o[n][3] *= al_b;
    }
    // O += P V: one 16-key step, d/8 column tiles (two per ldmatrix)
#pragma unroll
    for (int ks = 0; ks < 1; ++ks)
#pragma unroll
      for (int np = 0; np < kNT / 2; ++np) {
        uint32_t vb[4];
        const int key = kw + ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        ldsm_x4_t(vt + kv_swz<D, kTma>(key, 2 * np + (lane >> 4)), vb);
        mma16816<BF16>(o[2 * np], pf[ks], vb[0], vb[1]);
        mma16816<BF16>(o[2 * np + 1], pf[ks], vb[2], vb[3]);
      }
    __syncthreads();                       // this stage may be refilled next
  }
  cp_async_wait<0>();
  if (!ok) {
    // a wait gave up: let the copies still in flight land, then leave
    if (kTma && threadIdx.x == 0)
      for (int u = tile; u < tile + kStages && u < t1; ++u)   // issued: up to tile + kStages - 1
        mbar_wait_drain(&full[(u - t0) % kStages], ((u - t0) / kStages) & 1);
    return;
  }
  __syncthreads();

  // merge the four warps' partial results through shared memory
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  float *mrg = reinterpret_cast<float *>(dsm + L::kOffKV);   // [warp][row][D + 2]
  float *mw = mrg + warp * kRows * (D + 2);
#pragma unroll
  for (int n = 0; n < kNT; ++n) {
    mw[ra * (D + 2) + n * 8 + 2 * tq] = o[n][0];
    mw[ra * (D + 2) + n * 8 + 2 * tq + 1] = o[n][1];
    mw[rb * (D + 2) + n * 8 + 2 * tq] = o[n][2];
    mw[rb * (D + 2) + n * 8 + 2 * tq + 1] = o[n][3];
  }
  if (tq == 0) {
    mw[ra * (D + 2) + D] = m_a;
    mw[ra * (D + 2) + D + 1] = l_a;
    mw[rb * (D + 2) + D] = m_b;
    mw[rb * (D + 2) + D + 1] = l_b;
  }
  __syncthreads();
  // thread layout for the merge: 8 threads per row, D/8 columns each
  const int r = threadIdx.x >> 3, cg = threadIdx.x & 7;
  if (r < R) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) mx = fmaxf(mx, mrg[(w * kRows + r) * (D + 2) + D]);
    float wt[4], lsum = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float mw_ = mrg[(w * kRows + r) * (D + 2) + D];
      wt[w] = mx == -INFINITY ? 0.f : ex2(mw_ - mx);
      lsum += wt[w] * mrg[(w * kRows + r) * (D + 2) + D + 1];
    }
    const int qi = r / g, h = hk * g + r % g;
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const float lse_r = lsum > 0.f ? (mx + __log2f(lsum)) * 0.69314718055994531f : -INFINITY;
    const size_t orow = (static_cast<size_t>(b) * a.Nq + qi) * a.H + h;   // token-major row
    const size_t prow = (static_cast<size_t>(b) * a.H + h) * a.Nq + qi;   // [B, H, Nq] row
    if (a.splits == 1) {
      uint16_t *og = static_cast<uint16_t *>(a.o) + orow * D;
#pragma unroll
      for (int c = 0; c < D / 8; c += 2) {
        const int col = cg * (D / 8) + c;
        float x[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float acc = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w) acc += wt[w] * mrg[(w * kRows + r) * (D + 2) + col + e];
          x[e] = acc * inv;
        }
        *reinterpret_cast<uint32_t *>(og + col) = BF16 ? pack_bf16(x[0], x[1])
                                                        : pack_f16(x[0], x[1]);
      }
      if (cg == 0 && a.lse != nullptr) a.lse[prow] = lse_r;
    } else {
      const size_t part = static_cast<size_t>(split) * a.B * a.H * a.Nq + prow;
      float *wo = a.ws_o + part * D;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const int col = cg * (D / 8) + c;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) acc += wt[w] * mrg[(w * kRows + r) * (D + 2) + col];
        wo[col] = acc * inv;
      }
      if (cg == 0) a.ws_lse[part] = lse_r;
    }
  }
}

// Combine the splits' partial (O, lse) of each (b, h, query) row: one warp
// per row.  A split that saw no key has lse = -inf and weight 0.
template <int D, bool BF16>
__global__ void __launch_bounds__(128) merge_kernel(const DecodeArgs a) {
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int rows = a.B * a.H * a.Nq;
  if (row >= rows) return;
  const size_t stride = static_cast<size_t>(rows);
  // row = (b * H + h) * Nq + qi; sequence b wrote chunks 0 .. ceil(L_b / chunk) - 1
  const int Lb = __ldg(a.seqlens_k + row / (a.Nq * a.H));
  const int ns = Lb > 0 ? (Lb + a.chunk - 1) / a.chunk : 1;
  float mx = -INFINITY;
  for (int s = 0; s < ns; ++s) mx = fmaxf(mx, a.ws_lse[s * stride + row]);
  float acc[D / 32] = {}, z = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < ns; ++s) {
      const float w = __expf(a.ws_lse[s * stride + row] - mx);
      z += w;
      const float *po = a.ws_o + (s * stride + row) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) acc[c] += w * po[lane + 32 * c];
    }
  }
  // row = (b * H + h) * Nq + qi  ->  token-major output row (b, qi, h)
  const int qi = row % a.Nq, h = (row / a.Nq) % a.H, b = row / (a.Nq * a.H);
  uint16_t *og = static_cast<uint16_t *>(a.o) + ((static_cast<size_t>(b) * a.Nq + qi) * a.H + h) * D;
  const float inv = z > 0.f ? 1.f / z : 0.f;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    const float x = acc[c] * inv;
    og[lane + 32 * c] = BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x))
                             : __half_as_ushort(__float2half_rn(x));
  }
  if (lane == 0 && a.lse != nullptr) a.lse[row] = z > 0.f ? mx + logf(z) : -INFINITY;
}

template <int D, bool BF16, bool kTma>
attn_status_t launch_decode(const CUtensorMap &mk, const CUtensorMap &mv, DecodeArgs &a,
                            cudaStream_t s) {
  using L = DecSmem<D>;
  static std::once_flag once[kMaxDevices];
  static cudaError_t err[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::call_once(once[dev], [dev] {
    err[dev] = cudaFuncSetAttribute(decode_kernel<D, BF16, kTma>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  });
  if (err[dev] != cudaSuccess) return ATTN_ERR_LAUNCH;
  decode_kernel<D, BF16, kTma><<<dim3(a.splits, a.Hkv, a.B), kDecThreads, L::kBytes, s>>>(mk, mv, a);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  if (a.splits > 1) {
    const int rows = a.B * a.H * a.Nq;
    merge_kernel<D, BF16><<<(rows + 3) / 4, 128, 0, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

template <int D, bool BF16>
attn_status_t launch_decode_any(const CUtensorMap &mk, const CUtensorMap &mv, DecodeArgs &a,
                                cudaStream_t s) {
  return a.box_rows > 0 ? launch_decode<D, BF16, true>(mk, mv, a, s)
                        : launch_decode<D, BF16, false>(mk, mv, a, s);
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" attn_status_t attn_fwd_paged(const void *q, const void *k_cache, const void *v_cache,
                                        const int32_t *block_table, const int32_t *seqlens_k,
                                        void *o, float *lse, int B, int Nq, int H, int H_kv,
                                        int d, int page_size, int max_pages, int num_pages,
                                        int max_seqlen_k, float scale, int causal,
                                        attn_dtype_t dtype, int num_splits, void *stream) {
  if (!q || !k_cache || !v_cache || !block_table || !seqlens_k || !o) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Nq < 1 || H < 1 || H_kv < 1 || H % H_kv != 0 || page_size < 1 || max_pages < 1 ||
      num_pages < 1 || max_seqlen_k < 1 || num_splits < 0 || !std::isfinite(scale))
    return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  if ((H / H_kv) * Nq > kRows) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
    return ATTN_ERR_MISALIGNED;
  if ((lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seqlens_k) & 3u))
    return ATTN_ERR_MISALIGNED;
  if (static_cast<long long>(max_pages) * page_size < max_seqlen_k) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(num_pages) * page_size * H_kv * d > (1LL << 40) ||
      static_cast<long long>(B) * max_pages > (1LL << 31))
    return ATTN_ERR_TOO_LARGE;
  DeviceState *ds = nullptr;
  attn_status_t st = device_state(&ds);
  if (st != ATTN_OK) return st;
  // Chunk of keys per CTA.  Given num_splits, the longest sequence is cut
  // into that many chunks; otherwise the chunk is sized so that the key rows
  // of all sequences (at most B * max_seqlen_k) make about 16 CTAs per SM
  // (five to six waves of three), which evens out sequences of different
  // lengths while each CTA keeps enough tiles to run its copies ahead
  // (measured on the paged workload: 12 / 16 / 24 / 32 CTAs per SM give
  // 5340 / 5510 / 5125 / 5025 GB/s).
  const int tiles = (max_seqlen_k + kTileKeys - 1) / kTileKeys;
  long long chunk_tiles;
  if (num_splits > 0) {
    chunk_tiles = (tiles + num_splits - 1) / num_splits;
  } else {
    const long long work = static_cast<long long>(B) * H_kv * tiles;
    chunk_tiles = std::max<long long>(4, (work + 16LL * ds->num_sms - 1) / (16LL * ds->num_sms));
  }
  chunk_tiles = std::max<long long>(1, std::min<long long>(chunk_tiles, tiles));
  int splits = static_cast<int>((tiles + chunk_tiles - 1) / chunk_tiles);
  if (splits > 1024) {
    splits = 1024;
    chunk_tiles = (tiles + splits - 1) / splits;
    splits = static_cast<int>((tiles + chunk_tiles - 1) / chunk_tiles);
  }
  DecodeArgs a{};
  a.q = q; a.k = k_cache; a.v = v_cache; a.block_table = block_table; a.seqlens_k = seqlens_k;
  a.o = o; a.lse = lse;
  a.B = B; a.Nq = Nq; a.H = H; a.Hkv = H_kv; a.page_size = page_size; a.max_pages = max_pages;
  a.num_pages = num_pages; a.splits = splits;
  a.chunk = static_cast<int>(chunk_tiles * kTileKeys);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.causal = causal ? 1 : 0;
  if (splits > 1) {
    const size_t rows = static_cast<size_t>(B) * H * Nq;
    if ((st = ensure_split_workspace(ds, rows * splits * (d + 1) * sizeof(float))) != ATTN_OK)
      return st;
    a.ws_o = ds->split_ws;
    a.ws_lse = ds->split_ws + rows * splits * d;
  }
  a.status = ds->status;
  a.budget = wait_budget();
  // Tensor copies of the cache when a page splits into copies of 16, 32 or
  // 64 rows (64 % rows == 0 and page_size % rows == 0, so a tile's copies
  // never cross a page): the cache as a (d, H_kv, num_pages * page_size)
  // tensor, boxes of (64, 1, rows) with the 128-byte swizzle.  Otherwise the
  // rows are gathered with 16-byte copies.
  CUtensorMap mk{}, mv{};
  {
    int br = 64;
    while (br >= 16 && page_size % br != 0) br >>= 1;
    const long long rows = static_cast<long long>(num_pages) * page_size;
    a.box_rows = (br >= 16 && rows < (1LL << 31)) ? br : 0;
    if (a.box_rows > 0) {
      const CUtensorMapDataType dt =
          dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
      const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H_kv, (cuuint64_t)rows};
      const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H_kv * d * 2};
      const cuuint32_t box[3] = {64, 1, (cuuint32_t)a.box_rows};
      if ((st = encode_tiled(&mk, dt, 3, k_cache, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B)) != ATTN_OK ||
          (st = encode_tiled(&mv, dt, 3, v_cache, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B)) != ATTN_OK)
        return st;
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 128)
    return dtype == ATTN_BF16 ? launch_decode_any<128, true>(mk, mv, a, s)
                              : launch_decode_any<128, false>(mk, mv, a, s);
  return dtype == ATTN_BF16 ? launch_decode_any<64, true>(mk, mv, a, s)
                            : launch_decode_any<64, false>(mk, mv, a, s);
}
