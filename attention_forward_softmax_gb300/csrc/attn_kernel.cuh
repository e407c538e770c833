// attn_kernel.cuh -- fused attention forward for sm_103a.
//
// What it computes ("Fused attention kernel", wikillm concept card, Overview
// and Implementation sketch): for each query row, the running-softmax loop
// over key blocks -- new row max, rescale factor exp(m_old - m_new) applied to
// the running sum and the output, P = exp(S - m), O += P V -- then O / l and
// lse = m + log l.  Every key block is scored (the card's note on the
// printed loop bound), the rescale factor multiplies the OLD state (the
// card's note on the inverted factor).
//
// How it is laid out on the GPU (our design, not the card's Hopper one):
//  * one CTA per SM, persistent over work tiles; a work tile is 256 query
//    rows of one (sequence, head), split into two 128-row sub-tiles A and B;
//  * warp roles, 16-bit at d = 128 (320 threads):
//      warps 0-3  softmax warpgroup for sub-tile A (one thread per row)
//      warps 4-7  softmax warpgroup for sub-tile B
//      warp  8    MMA issuer (one thread) + TMEM allocation
//      warp  9    TMA producer (one thread)
//  * warp roles, e4m3 and 16-bit at d = 64 (352 threads), where S is free
//    as soon as the softmax has read it:
//      warps 0-7  softmax, one thread per row (sub-tile A, then B)
//      warp  8    MMA issuer of sub-tile A (S_A and O_A) + TMEM allocation
//      warp  9    TMA producer
//      warp 10    MMA issuer of sub-tile B
//  * Q sub-tiles stay in shared memory for the whole tile; K and V tiles of
//    128 keys stream through a ring of NS slots (K_0, V_0, K_1, V_1, ...);
//  * TMEM (512 columns): S_A [0,128), S_B [128,256), O_A, O_B after them;
//    16-bit P is written back over the first columns of its S at d = 128
//    and gets its own columns after O at d = 64; e4m3 P goes to one
//    shared-memory tile per sub-tile;
//  * 16-bit tensor-core order per key block j at d = 128:  S_A(j), O_B += P_B(j-1)
//    V_{j-1}, S_B(j), O_A += P_A(j) V_j -- so each softmax warpgroup works
//    while the tensor core serves the other sub-tile.  A commit after S_X(j)
//    also covers the earlier O_X update, so when softmax X sees S_X(j) ready
//    its O is current and it may rescale O in place;
//  * e4m3 and d = 64: S_X(j+1) is issued as soon as softmax X has read
//    S_X(j) into registers, by the issuing thread of sub-tile X;
//    O_X += P_X(j) V_j waits for P, and the softmax waits for that update
//    before it rescales O_X or rewrites P;
//  * the output is rescaled only when a row max grows by more than
//    kRescaleThresh (log2 units); otherwise the stale max is kept, which is
//    exact after the final division by l;
//  * e4m3: the V descale of each key block is folded into P (stored as
//    e4m3(p * w)) with w kept in [1, 8] by re-basing the output's unit,
//    which rescales O like a grown row max;
//  * every mbarrier wait is bounded (clock64 budget): on expiry the kernel
//    records ATTN_ERR_TIMEOUT in the status word, drains its own copies and
//    MMAs, frees TMEM and returns.
#pragma once

#include "ptx.cuh"

namespace attn {

enum class Elem : int { BF16 = 0, F16 = 1, E4M3 = 2 };

struct Params {
  void *o;                  // output [B,N,H,d] or [T,H,d] (bf16/f16; bf16 for e4m3 inputs)
  float *lse;               // [B,H,N] or [H,T]; may be null
  const int *cu_seqlens;    // varlen: [nseq+1]
  const int2 *tiles;        // varlen: (sequence, query-tile) in schedule order
  const int *num_entries;   // varlen: number of valid entries in `tiles`
  int B;                    // dense: batch; varlen: number of sequences
  int H;                    // query (and output) heads
  int grp;                  // query heads per K/V head (H / H_kv)
  int N;                    // dense: sequence length; varlen: max sequence length
  int T;                    // varlen: total tokens
  int num_tiles;            // dense: exact count; varlen: upper bound
  int causal;
  float scale_log2;         // scale * log2(e)
  const float *dq, *dk, *dv;  // e4m3: per-block descales [B,H,nblk] (Q), [B,H_kv,nblk] (K, V)
  int nblk;
  int d_out;                // head size of the tensors (e4m3: 64 runs the 128-column layout
                            // with the upper 64 columns of Q, K, V zero-filled by the copies)
  long long wait_budget;
  int *status;
  const float *bias;        // additive score bias (kBias): bias[b*sb + h*sh + row*sr + key]
  long long bias_sb, bias_sh, bias_sr;
  // Dense, non-causal: work items from split_from on (when >= 0) are the
  // two key halves of the last tiles, so that the final wave of a
  // persistent grid is not left mostly idle.  Item split_from + u is half
  // u & 1 of tile split_from + u / 2; it writes O / l (fp32) and its lse to
  // part u of part_o [parts][256][D] and part_lse [parts][256].
  int split_from;
  float *part_o, *part_lse;
};

template <int D_, Elem E_, bool Varlen_, bool Bias_ = false>
struct Cfg {
  static constexpr int D = D_;
  static constexpr Elem E = E_;
  static constexpr bool kVarlen = Varlen_;
  // an fp32 bias added to the scores (16-bit, dense layout)
  static constexpr bool kBias = Bias_;
  static_assert(!Bias_ || (E_ != Elem::E4M3 && !Varlen_), "bias: 16-bit dense only");
  static constexpr bool kFp8 = (E_ == Elem::E4M3);
  static constexpr int kElt = kFp8 ? 1 : 2;
  static constexpr int BM = 128;                       // rows per sub-tile
  static constexpr int BN = 128;                       // keys per K/V tile
  static constexpr int kRowBytes = D * kElt;           // one row of a tile
  static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte swizzle rows");
  static constexpr int kChunks = kRowBytes / 128;      // 128-byte column chunks per row
  static constexpr int kChunkElems = 128 / kElt;
  static constexpr int kChunkBytes = 128 * 128;        // 128 rows x 128 bytes
  static constexpr int kTileBytes = 128 * kRowBytes;   // one Q sub-tile / K or V tile
  static constexpr int kSmemBudget = 224 * 1024;
  // K/V ring: the largest power of two of tiles (at most 8) that fits beside
  // the two Q sub-tiles and, for e4m3, the two P tiles
  static constexpr int kRingFit =
      (kSmemBudget - 2 * kTileBytes - 2 * (kFp8 ? 2 * 128 * 128 : 0)) / kTileBytes;
  static constexpr int NS = kRingFit >= 8 ? 8 : (kRingFit >= 4 ? 4 : 2);
  static_assert(NS >= 3, "K/V ring too small");
  static_assert((NS & (NS - 1)) == 0, "K/V ring size must be a power of two");
  // K and V tiles alternate through the ring, so with an even ring a slot
  // always holds K or always V, and every issuer that waits on a slot's full
  // barrier waits for each of its phases in order.  With an odd ring one
  // issuer could reach a slot's next use while its other use was still
  // pending, and its parity wait would pass a phase early.
  static_assert(NS % 2 == 0, "K/V ring size must be even");
  // MMA shapes.  Each instruction consumes 32 bytes of K per row.
  static constexpr int kKStep = 32 / kElt;             // 16 (16-bit) or 32 (e4m3)
  static constexpr int kQKSteps = kRowBytes / 32;
  static constexpr int kPVSteps = BN / kKStep;
  static constexpr uint32_t kFmt = (E_ == Elem::BF16) ? 1u : 0u;
  static constexpr uint32_t kIdescQK = idesc_make(kFmt, 128, BN, false, false);
  static constexpr uint32_t kIdescPV = idesc_make(kFmt, 128, D, false, true);
  // TMEM columns
  static constexpr uint32_t kColS = 128;              // S_X starts at column x * kColS
  static constexpr uint32_t kColO0 = 256;
  static constexpr int kPCols = BN * kElt / 4;         // 64 (16-bit P) or 32 (e4m3 P)
  // Output rescale threshold in log2 units: p may grow to 2^thresh between
  // rescales.  16-bit P: 2^8.  e4m3 P is stored as p * w with the prescale
  // w <= kP8Scale: at most 2^5.75 * 8 = 430, below the e4m3 maximum 448.  (A
  // larger prescale buys nothing in accuracy and a lower threshold; with
  // outlier keys a 32-row warp then rescales O on a quarter of its key
  // blocks instead of a twelfth.)
  static constexpr float kP8Scale = 8.f;
  static constexpr float kRescaleThresh = kFp8 ? 5.75f : 8.0f;
  // e4m3: P goes to shared memory (one 128 x 128-byte tile per sub-tile, the
  // 128-byte-swizzled K-major layout), so S can be overwritten as soon as the
  // softmax has read it; 16-bit P stays in TMEM over S.
  static constexpr bool kSmemP = kFp8;
  static constexpr int kPTileBytes = kSmemP ? 128 * 128 : 0;
  // P tiles per sub-tile: two for e4m3, so the exponentials of a block do
  // not wait for the O update that reads the previous block's P
  static constexpr int kPBufs = kSmemP ? 2 : 1;
  // 16-bit at d = 64: O_A and O_B take only 128 TMEM columns, so P gets its
  // own 64 columns per sub-tile after them and S is free once it is read,
  // as in the e4m3 path (P in TMEM rather than shared memory).
  static constexpr bool kSepP = !kFp8 && D == 64;
  static constexpr uint32_t kColP0 = 256 + 2 * D;        // kSepP: P_X at kColP0 + 64 x
  static constexpr bool kDual = kSmemP || kSepP;         // one MMA issuer per sub-tile
  // softmax warps: one thread per query row of the two sub-tiles
  static constexpr int kSoftmaxWarps = 8;
  static constexpr int kWarpMMA = kSoftmaxWarps;       // MMA issuer (kDual: of sub-tile A) + TMEM allocation
  static constexpr int kWarpTMA = kSoftmaxWarps + 1;   // TMA producer
  static constexpr int kWarpPV = kSoftmaxWarps + 2;    // kDual: MMA issuer of sub-tile B
  static constexpr int kThreads = 32 * (kSoftmaxWarps + 2 + (kDual ? 1 : 0));
  // arrivals per phase on the barriers the softmax signals: one per softmax
  // thread of the sub-tile
  static constexpr int kSoftArrive = 32 * kSoftmaxWarps / 2;
  // shared memory layout (offsets from the 1024-aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = 2 * kTileBytes;
  static constexpr int kOffP = kOffKV + NS * kTileBytes;
  static constexpr int kOffBar = kOffP + 2 * kPBufs * kPTileBytes;
  static constexpr int kNumBars = 2 + 2 * NS + 17;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 64 + 1024 /* alignment slack */ + 1024 /* guard */;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA exceeded");
};

struct TileInfo {
  int b;          // dense batch index / varlen sequence index
  int h;          // query head
  int hk;         // its K/V head
  int qt;         // query tile (256 rows) within the sequence
  int L;          // sequence length
  int start;      // first token of the sequence in the packed / flattened rows
  int nA, nB;     // key tiles processed by sub-tiles A and B
  int kb0;        // first key tile (a key half of a split tile: nkv / 2)
  int part;       // split partial written by this item, or -1
};

template <class C>
__device__ __forceinline__ bool get_tile(const Params &p, int t, int num_tiles, TileInfo &ti) {
  if (t >= num_tiles) return false;
  int half = -1;
  if constexpr (!C::kVarlen) {
    if (p.split_from >= 0 && t >= p.split_from) {   // a key half of a split tile
      half = (t - p.split_from) & 1;
      ti.part = t - p.split_from;
      t = p.split_from + ((t - p.split_from) >> 1);
    }
    const int nqt = (p.N + 255) / 256;
    const int BH = p.B * p.H;
    int bh;
    if (p.causal) {   // heaviest query tiles first (longest-processing-time order)
      ti.qt = nqt - 1 - t / BH;
      bh = t % BH;
    } else {          // neighbouring CTAs share one head's K/V in L2
      bh = t / nqt;
      ti.qt = t % nqt;
    }
    ti.b = bh / p.H;
    ti.h = bh % p.H;
    ti.L = p.N;
    ti.start = ti.b * p.N;
  } else {
    // Heads outermost (t = h * entries + e): the CTAs running at one time
    // share one head, whose K/V over all sequences stays in L2; within a
    // head the list is heaviest first.
    const int ne = num_tiles / p.H;
    const int2 e = p.tiles[t % ne];
    ti.h = t / ne;
    ti.b = e.x;
    ti.qt = e.y;
    ti.start = p.cu_seqlens[e.x];
    ti.L = p.cu_seqlens[e.x + 1] - ti.start;
  }
  ti.hk = ti.h / p.grp;
  const int nkv = (ti.L + 127) / 128;
  if (p.causal) {
    ti.nA = min(2 * ti.qt + 1, nkv);
    ti.nB = (ti.qt * 256 + 128 < ti.L) ? min(2 * ti.qt + 2, nkv) : ti.nA;
  } else {
    ti.nA = nkv;
    ti.nB = nkv;
  }
  ti.kb0 = 0;
  if (half < 0) {
    ti.part = -1;
  } else {
    ti.kb0 = half ? nkv / 2 : 0;
    ti.nA = ti.nB = half ? nkv - nkv / 2 : nkv / 2;
  }
  return true;
}

template <class C>
__device__ __forceinline__ int tile_count(const Params &p) {
  if constexpr (C::kVarlen) {
    return min(p.num_tiles, __ldg(p.num_entries) * p.H);
  } else {
    return p.num_tiles;
  }
}

// A key half of a split tile: this thread's row of O / l in fp32 and its lse
// (natural log, over this half's keys) go to the item's partial.
template <class C>
__device__ __forceinline__ void store_partial_row(const Params &p, const TileInfo &ti, int x,
                                                  int r_in, uint32_t tO, float inv_l,
                                                  float m_run, float l_run) {
  const bool valid = ti.qt * 256 + x * 128 + r_in < ti.L;
  const size_t prow = static_cast<size_t>(ti.part) * 256 + x * 128 + r_in;
  float *dst = p.part_o + prow * C::D;
#pragma unroll 1
  for (int c = 0; c < C::D / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(tO + c * 32, o);
    if (valid) {
      float4 *d4 = reinterpret_cast<float4 *>(dst + c * 32);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        d4[i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                            __uint_as_float(o[4 * i + 2]) * inv_l,
                            __uint_as_float(o[4 * i + 3]) * inv_l);
    }
  }
  if (valid) p.part_lse[prow] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
}

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem + C::kOffQ;
  uint8_t *sKV = smem + C::kOffKV;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *bar_q_full = bars + 0;
  uint64_t *bar_q_empty = bars + 1;
  uint64_t *bar_kv_full = bars + 2;
  uint64_t *bar_kv_empty = bars + 2 + C::NS;
  uint64_t *bar_s_full = bars + 2 + 2 * C::NS;     // [2]
  uint64_t *bar_p_full = bar_s_full + 2;           // [2]
  uint64_t *bar_o_final = bar_s_full + 4;          // [2]
  uint64_t *bar_o_free = bar_s_full + 6;           // [2]
  uint64_t *bar_drain = bar_s_full + 8;
  uint64_t *bar_s_free = bar_s_full + 9;           // [2] e4m3: softmax has read S
  uint64_t *bar_o_done = bar_s_full + 11;          // [2] e4m3, d = 64: an O update completed
  // e4m3, second P tile of each sub-tile: its P-full and O-done barriers
  uint64_t *bar_p_full1 = bar_s_full + 13;         // [2]
  uint64_t *bar_o_done1 = bar_s_full + 15;         // [2]
  // the barriers of P tile b of sub-tile x
  auto p_full_bar = [&](int x, int b) { return b ? &bar_p_full1[x] : &bar_p_full[x]; };
  auto o_done_bar = [&](int x, int b) { return b ? &bar_o_done1[x] : &bar_o_done[x]; };
  uint8_t *sP = smem + C::kOffP;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 1);
    // dual issuers: both release the Q buffer and every K/V slot
    mbar_init(bar_q_empty, C::kDual ? 2 : 1);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&bar_kv_full[i], 1);
      mbar_init(&bar_kv_empty[i], C::kDual ? 2 : 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar_s_full[x], 1);
      mbar_init(&bar_p_full[x], C::kSoftArrive);
      mbar_init(&bar_o_final[x], 1);
      mbar_init(&bar_o_free[x], C::kSoftArrive);
    }
    mbar_init(bar_drain, C::kDual ? 2 : 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar_s_free[x], C::kSoftArrive);
      mbar_init(&bar_o_done[x], 1);
      mbar_init(&bar_p_full1[x], C::kSoftArrive);
      mbar_init(&bar_o_done1[x], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kWarpMMA) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  if (warp == C::kWarpTMA && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const WaitCtl wc{abort_flag, p.status, p.wait_budget};
  const int num_tiles = tile_count<C>(p);
  if (warp == C::kWarpTMA) {
    // ------------------------------------------------------------------
    // TMA producer
    // ------------------------------------------------------------------
    if (lane == 0) {
      // Q is read once per tile; K and V are read again by the CTAs that
      // work on the other query tiles of the head
      const uint64_t pol_q = l2_policy_evict_first(), pol_kv = l2_policy_evict_last();
      int kv_pos = 0, tcount = 0, q_issued = 0;
      bool ok = true;
      TileInfo ti;
      for (int t = blockIdx.x; ok && get_tile<C>(p, t, num_tiles, ti); t += gridDim.x, ++tcount) {
        if (!mbar_wait(bar_q_empty, (tcount & 1) ^ 1, wc)) { ok = false; break; }
        mbar_arrive_expect_tx(bar_q_full, 2 * C::kTileBytes);
        ++q_issued;
        for (int x = 0; x < 2; ++x) {
          const int row = ti.qt * 256 + x * 128;
          for (int c = 0; c < C::kChunks; ++c) {
            uint8_t *dst = sQ + x * C::kTileBytes + c * C::kChunkBytes;
            if constexpr (C::kVarlen)
              tma_load_3d_hint(dst, &tmQ, bar_q_full, c * C::kChunkElems, ti.h, ti.start + row,
                               pol_q);
            else
              tma_load_4d_hint(dst, &tmQ, bar_q_full, c * C::kChunkElems, ti.h, row, ti.b, pol_q);
          }
        }
        for (int j = 0; ok && j < ti.nB; ++j) {
          for (int kv = 0; kv < 2; ++kv, ++kv_pos) {
            const int slot = kv_pos % C::NS;
            const int round = kv_pos / C::NS;
            if (!mbar_wait(&bar_kv_empty[slot], (round & 1) ^ 1, wc)) { ok = false; break; }
            mbar_arrive_expect_tx(&bar_kv_full[slot], C::kTileBytes);
            const CUtensorMap *map = kv == 0 ? &tmK : &tmV;
            for (int c = 0; c < C::kChunks; ++c) {
              uint8_t *dst = sKV + slot * C::kTileBytes + c * C::kChunkBytes;
              if constexpr (C::kVarlen)
                tma_load_3d_hint(dst, map, &bar_kv_full[slot], c * C::kChunkElems, ti.hk,
                                 ti.start + (ti.kb0 + j) * 128, pol_kv);
              else
                tma_load_4d_hint(dst, map, &bar_kv_full[slot], c * C::kChunkElems, ti.hk,
                                 (ti.kb0 + j) * 128, ti.b, pol_kv);
            }
          }
        }
      }
      if (!ok) {
        // Drain: wait (bounded) for the last copy issued into every slot and
        // for the last Q copy, so no copy lands after the CTA has exited.
        for (int i = 0; i < C::NS && i < kv_pos; ++i) {
          const int pos = kv_pos - 1 - i;
          mbar_wait_drain(&bar_kv_full[pos % C::NS], (pos / C::NS) & 1);
        }
        if (q_issued > 0) mbar_wait_drain(bar_q_full, (q_issued - 1) & 1);
      }
    }
  } else if (warp == C::kWarpMMA || (C::kDual && warp == C::kWarpPV)) {
    // ------------------------------------------------------------------
    // MMA issuer(s)
    // ------------------------------------------------------------------
    if (lane == 0) {
      // Shared-memory descriptors are built once.  Per MMA only a constant
      // (the byte offset >> 4) is added to the low word, whose start-address
      // field [0,14) has room for any shared-memory offset, so no carry
      // reaches the other fields: one integer add per operand per MMA.
      const uint64_t q0 = sdesc_sw128(smem_addr(sQ), 16, 1024);
      const uint64_t k0 = sdesc_sw128(smem_addr(sKV), 16, 1024);
      const uint64_t v0 = sdesc_sw128(smem_addr(sKV), C::kChunkBytes, 1024);
      const uint32_t q_lo = static_cast<uint32_t>(q0), q_hi = static_cast<uint32_t>(q0 >> 32);
      const uint32_t k_lo = static_cast<uint32_t>(k0), k_hi = static_cast<uint32_t>(k0 >> 32);
      const uint32_t v_lo = static_cast<uint32_t>(v0), v_hi = static_cast<uint32_t>(v0 >> 32);
      auto desc = [](uint32_t lo, uint32_t hi) { return (static_cast<uint64_t>(hi) << 32) | lo; };
      unsigned kv_pos = 0;
      int tcount = 0;
      unsigned p_cnt[2] = {0, 0};
      bool ok = true;
      TileInfo ti;

      // S_X = Q_X K^T  (K tile at ring position pos)
      auto issue_qk = [&](int x, unsigned pos) {
        const uint32_t qa = q_lo + static_cast<uint32_t>(x * (C::kTileBytes >> 4));
        const uint32_t ka = k_lo + (pos & (C::NS - 1)) * (C::kTileBytes >> 4);
        const uint32_t d = tmem + x * C::kColS;
#pragma unroll
        for (int s = 0; s < C::kQKSteps; ++s) {
          const uint32_t off = ((s / 4) * C::kChunkBytes + (s % 4) * 32) >> 4;
          if constexpr (C::kFp8)
            mma_f8_ss(d, desc(qa + off, q_hi), desc(ka + off, k_hi), C::kIdescQK, s > 0);
          else
            mma_f16_ss(d, desc(qa + off, q_hi), desc(ka + off, k_hi), C::kIdescQK, s > 0);
        }
      };
      // O_X (+)= P_X V  (V tile at ring position pos)
      auto issue_pv = [&](int x, unsigned pos, bool accumulate) {
        const uint32_t va = v_lo + (pos & (C::NS - 1)) * (C::kTileBytes >> 4);
        const uint32_t d = tmem + C::kColO0 + x * C::D;
        const uint32_t pa = tmem + (C::kSepP ? C::kColP0 + x * 64 : x * C::kColS);
        if constexpr (C::kFp8)
          mma_f8_ts(d, pa, desc(va, v_hi), C::kIdescPV, accumulate);
        else
          mma_f16_ts(d, pa, desc(va, v_hi), C::kIdescPV, accumulate);
#pragma unroll
        for (int s = 1; s < C::kPVSteps; ++s) {
          const uint32_t off = (s * C::kKStep * 128) >> 4;
          if constexpr (C::kFp8)
            mma_f8_ts(d, pa + s * 8, desc(va + off, v_hi), C::kIdescPV, 1);
          else
            mma_f16_ts(d, pa + s * 8, desc(va + off, v_hi), C::kIdescPV, 1);
        }
      };
      // O_X (+)= P_X V with P_X in shared memory (e4m3 path)
      const uint64_t p0d = sdesc_sw128(smem_addr(sP), 16, 1024);
      const uint32_t p_lo = static_cast<uint32_t>(p0d), p_hi = static_cast<uint32_t>(p0d >> 32);
      auto issue_pv_smem = [&](int x, int pb, unsigned pos, bool accumulate) {
        const uint32_t va = v_lo + (pos & (C::NS - 1)) * (C::kTileBytes >> 4);
        const uint32_t pa =
            p_lo + static_cast<uint32_t>((x * C::kPBufs + pb) * (C::kPTileBytes >> 4));
        const uint32_t d = tmem + C::kColO0 + x * C::D;
        mma_f8_ss(d, desc(pa, p_hi), desc(va, v_hi), C::kIdescPV, accumulate);
#pragma unroll
        for (int s = 1; s < C::kPVSteps; ++s)
          mma_f8_ss(d, desc(pa + ((s * 32) >> 4), p_hi),
                    desc(va + ((s * C::kKStep * 128) >> 4), v_hi), C::kIdescPV, 1);
      };
      unsigned qk_cnt[2] = {0, 0};
      // e4m3: QK_X may overwrite S_X once the softmax has read the previous S_X
      auto wait_s_free = [&](int x) {
        if (qk_cnt[x] > 0 && !mbar_wait(&bar_s_free[x], (qk_cnt[x] - 1) & 1, wc)) return false;
        ++qk_cnt[x];
        tc_fence_after();
        return true;
      };
      auto wait_kv = [&](unsigned pos) {
        if (!mbar_wait(&bar_kv_full[pos & (C::NS - 1)], (pos / C::NS) & 1, wc)) return false;
        tc_fence_after();
        return true;
      };
      // P tile c of sub-tile x (counted over the whole run) is buffer
      // c mod kPBufs, whose barrier completes for it for the (c / kPBufs)-th
      // time
      auto wait_p = [&](int x) {
        const unsigned c = p_cnt[x];
        if (!mbar_wait(p_full_bar(x, c % C::kPBufs), (c / C::kPBufs) & 1, wc)) return false;
        ++p_cnt[x];
        tc_fence_after();
        return true;
      };

      if constexpr (C::kDual) {
        // e4m3, and 16-bit at d = 64: one issuing thread per sub-tile.  Warp
        // kWarpMMA serves sub-tile A, warp kWarpPV sub-tile B; each issues
        // S_X(j+1) = Q_X K_{j+1}^T as soon as softmax X has read S_X(j), then
        // O_X += P_X(j) V_j as soon as P_X(j) is written (shared memory for
        // e4m3, its own TMEM columns for 16-bit), so neither sub-tile's
        // products wait for the other's softmax.  Both issuers release every
        // K/V slot and the Q buffer (two arrivals each); the one with fewer
        // key tiles (A, on the causal diagonal) still waits for the copies
        // of the tiles it skips, so it sees every slot's phases in order.
        const int x = warp == C::kWarpMMA ? 0 : 1;
        for (int t = blockIdx.x; ok && get_tile<C>(p, t, num_tiles, ti); t += gridDim.x, ++tcount) {
          const int nX = x == 0 ? ti.nA : ti.nB, nB = ti.nB;
          if (!mbar_wait(bar_q_full, tcount & 1, wc)) { ok = false; break; }
          tc_fence_after();
          // S_X(0)
          if (!wait_kv(kv_pos) || !wait_s_free(x)) { ok = false; break; }
          issue_qk(x, kv_pos);
          mma_commit(&bar_s_full[x]);
          mma_commit(&bar_kv_empty[kv_pos & (C::NS - 1)]);
          if (nX == 1) mma_commit(bar_q_empty);
          for (int j = 0; j < nX; ++j) {
            if (j + 1 < nX) {   // S_X(j+1)
              const unsigned pk = kv_pos + 2 * (j + 1);
              if (!wait_kv(pk) || !wait_s_free(x)) { ok = false; break; }
              issue_qk(x, pk);
              mma_commit(&bar_s_full[x]);
              mma_commit(&bar_kv_empty[pk & (C::NS - 1)]);
              if (j + 2 == nX) mma_commit(bar_q_empty);
            }
            // O_X (+)= P_X(j) V_j
            const unsigned pv = kv_pos + 2 * j + 1;
            if (!wait_kv(pv)) { ok = false; break; }
            if (j == 0 && !mbar_wait(&bar_o_free[x], (tcount & 1) ^ 1, wc)) { ok = false; break; }
            const int pb = static_cast<int>(p_cnt[x] % C::kPBufs);
            if (!wait_p(x)) { ok = false; break; }
            if constexpr (C::kSmemP) issue_pv_smem(x, pb, pv, j > 0);
            else issue_pv(x, pv, j > 0);
            mma_commit(o_done_bar(x, pb));
            if (j == nX - 1) mma_commit(&bar_o_final[x]);
            mma_commit(&bar_kv_empty[pv & (C::NS - 1)]);
          }
          if (!ok) break;
          // key tiles of the other sub-tile only
          for (int j = nX; j < nB; ++j) {
            for (int u = 0; u < 2; ++u) {
              const unsigned pos = kv_pos + 2 * j + u;
              if (!wait_kv(pos)) { ok = false; break; }
              mma_commit(&bar_kv_empty[pos & (C::NS - 1)]);
            }
            if (!ok) break;
          }
          kv_pos += 2 * nB;
        }
      } else
      for (int t = blockIdx.x; ok && get_tile<C>(p, t, num_tiles, ti); t += gridDim.x, ++tcount) {
        const int nA = ti.nA, nB = ti.nB;
        if (!mbar_wait(bar_q_full, tcount & 1, wc)) { ok = false; break; }
        tc_fence_after();
        for (int j = 0; j < nB; ++j) {
          const unsigned pk = kv_pos + 2 * j, pv = pk + 1;
          if (!wait_kv(pk)) { ok = false; break; }
          if (j < nA) {
            issue_qk(0, pk);
            mma_commit(&bar_s_full[0]);
          }
          if (j >= 1) {   // O_B (+)= P_B(j-1) V_{j-1}
            if (!wait_p(1)) { ok = false; break; }
            if (j - 1 == 0) {
              if (!mbar_wait(&bar_o_free[1], (tcount & 1) ^ 1, wc)) { ok = false; break; }
              tc_fence_after();
            }
            if (j - 1 >= nA && !wait_kv(pv - 2)) { ok = false; break; }
            issue_pv(1, pv - 2, j - 1 > 0);
            mma_commit(&bar_kv_empty[(pv - 2) & (C::NS - 1)]);
          }
          issue_qk(1, pk);
          mma_commit(&bar_s_full[1]);
          mma_commit(&bar_kv_empty[pk & (C::NS - 1)]);
          if (j == nB - 1) mma_commit(bar_q_empty);
          if (j < nA) {   // O_A (+)= P_A(j) V_j
            if (!wait_p(0)) { ok = false; break; }
            if (j == 0) {
              if (!mbar_wait(&bar_o_free[0], (tcount & 1) ^ 1, wc)) { ok = false; break; }
              tc_fence_after();
            }
            if (!wait_kv(pv)) { ok = false; break; }
            issue_pv(0, pv, j > 0);
            if (j == nA - 1) mma_commit(&bar_o_final[0]);
          }
        }
        if (!ok) break;
        {   // O_B (+)= P_B(nB-1) V_{nB-1}
          const int j = nB - 1;
          const unsigned pv = kv_pos + 2 * j + 1;
          if (!wait_p(1)) { ok = false; break; }
          if (j == 0) {
            if (!mbar_wait(&bar_o_free[1], (tcount & 1) ^ 1, wc)) { ok = false; break; }
            tc_fence_after();
          }
          if (j >= nA && !wait_kv(pv)) { ok = false; break; }
          issue_pv(1, pv, j > 0);
          mma_commit(&bar_o_final[1]);
          mma_commit(&bar_kv_empty[pv & (C::NS - 1)]);
        }
        kv_pos += 2 * nB;
      }
      // Drain every MMA this thread issued before TMEM is released.
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
    __syncwarp();
  } else if constexpr (C::kFp8) {
    // ------------------------------------------------------------------
    // e4m3 softmax, one thread per query row: warp w serves sub-tile
    // x = w >> 2 and TMEM lane quarter w & 3.  The thread reads its whole
    // 128-key score row, writes its 128-byte row of the P tile (16-byte
    // chunk c at c ^ (row & 7): the 128-byte swizzle) and owns its row of O.
    // ------------------------------------------------------------------
    const int x = warp >> 2;
    const int wq = warp & 3;
    const int r_in = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + x * C::kColS;
    const uint32_t tO = tmem + lane_base + C::kColO0 + x * C::D;
    const uint32_t p_row0 = smem_addr(sP) + x * C::kPBufs * C::kPTileBytes + r_in * 128;
    int s_cnt = 0, tcount = 0;
    unsigned pstore_cnt = 0;
    bool ok = true;
    TileInfo ti;
    for (int t = blockIdx.x; ok && get_tile<C>(p, t, num_tiles, ti); t += gridDim.x, ++tcount) {
      const int nX = x == 0 ? ti.nA : ti.nB;
      const int row0 = ti.qt * 256 + x * 128;
      const int row = row0 + r_in;
      float m_run = -INFINITY;                          // running max, log2 units
      float l_run = 0.f;
      // Per-block descales of this (b, h).  The V descale dv_j of key block
      // j is folded into P: it is stored as p * w, w = kP8Scale * dv_j / R,
      // so O accumulates in units of R / kP8Scale.  R starts at the largest
      // dv of the (b, h); when w would leave [kP8Scale / 8, kP8Scale] (a
      // block whose scale is far below R, or above it after such a change),
      // R is re-based to dv_j and O rescaled with it, like the row maximum.
      const size_t dbase = (static_cast<size_t>(ti.b) * p.H + ti.h) * p.nblk;
      const size_t kvbase = (static_cast<size_t>(ti.b) * (p.H / p.grp) + ti.hk) * p.nblk;
      const float dq_s = __ldg(p.dq + dbase + (row0 >> 7));
      const float *dk_row = p.dk + kvbase;
      const float *dv_row = p.dv + kvbase;
      float dvm = 0.f;
      for (int i = lane; i < (ti.L + 127) / 128; i += 32) dvm = fmaxf(dvm, __ldg(dv_row + i));
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) dvm = fmaxf(dvm, __shfl_xor_sync(0xffffffffu, dvm, m));
      float r_unit = C::kP8Scale / dvm;                 // kP8Scale / R
      float dk_next = __ldg(dk_row + ti.kb0), dv_next = __ldg(dv_row + ti.kb0);
      for (int j = 0; j < nX; ++j) {
        if (!__all_sync(0xffffffffu, mbar_wait(&bar_s_full[x], s_cnt & 1, wc))) { ok = false; break; }
        ++s_cnt;
        tc_fence_after();
        uint32_t sv[128];
        float mx_ld;                      // row maximum, from the load itself
        tmem_ld128_max(tS, sv, mx_ld);
        // S is in registers: the tensor core may overwrite it
        tc_fence_before();
        mbar_arrive(&bar_s_free[x]);
        const float cs = p.scale_log2 * dq_s * dk_next;   // log2 units per raw score
        float pw = dv_next * r_unit;
        float unit_f = 1.f;                                 // O rescale from re-basing R
        // (the upper test has a little slack so that the block that sets R
        // does not re-base through rounding; p * w stays below 448 up to
        // w = 8.3)
        if (pw < C::kP8Scale * 0.125f || pw > C::kP8Scale * 1.03125f) {   // uniform over (b, h)
          unit_f = C::kP8Scale / pw;
          r_unit = C::kP8Scale / dv_next;
          pw = C::kP8Scale;
        }
        if (j + 1 < nX) {
          dk_next = __ldg(dk_row + ti.kb0 + j + 1);
          dv_next = __ldg(dv_row + ti.kb0 + j + 1);
        }
        const int kbase = (ti.kb0 + j) * 128;
        if ((kbase + 128 > ti.L) || (p.causal && kbase + 127 > row0)) {
          const int lim = p.causal ? min(ti.L, row + 1) : ti.L;   // keys < lim allowed
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (kbase + i >= lim) sv[i] = __float_as_uint(-INFINITY);
          // row maximum of the masked row: four independent three-input chains
          float mx4[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t *sc = sv + 32 * c;
            float m = fmaxf(__uint_as_float(sc[0]), __uint_as_float(sc[1]));
#pragma unroll
            for (int i = 2; i < 32; i += 2) m = fmax3(m, __uint_as_float(sc[i]), __uint_as_float(sc[i + 1]));
            mx4[c] = m;
          }
          mx_ld = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        }
        const float m_tile = mx_ld * cs;
        const float m_new = fmaxf(m_run, m_tile);
        const bool resc = m_new > m_run + C::kRescaleThresh;
        float alpha = 1.f;
        if (resc) {
          alpha = ex2(m_run - m_new);    // 0 when m_run = -inf
          l_run *= alpha;
          m_run = m_new;
        }
        // P tile pc (of this sub-tile, counted over the run) goes to buffer
        // pb = pc mod 2, once the O update that read tile pc - 2 from it is
        // complete
        const unsigned pc = pstore_cnt++;
        const int pb = static_cast<int>(pc & 1);
        if (pc >= 2 &&
            !__all_sync(0xffffffffu, mbar_wait(o_done_bar(x, pb), ((pc >> 1) - 1) & 1, wc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t p_row = p_row0 + pb * C::kPTileBytes;
        // stored value p * pw = 2^(s*cs - m + log2 pw), the prescale folded
        // into the exponent; row sums of the stored values in packed fp32,
        // divided by pw once per key block
        const float lpw = __log2f(fmaxf(pw, 1e-30f));
        const float mb = m_run - lpw;
        float ra[4] = {0.f, 0.f, 0.f, 0.f}, rb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t *sr = sv + 16 * c;
          uint32_t pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float x0, x1, x2, x3;
            ffma2(x0, x1, __uint_as_float(sr[4 * i]), __uint_as_float(sr[4 * i + 1]), cs, cs, -mb,
                  -mb);
            ffma2(x2, x3, __uint_as_float(sr[4 * i + 2]), __uint_as_float(sr[4 * i + 3]), cs, cs,
                  -mb, -mb);
            const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
            fadd2(ra[i], rb[i], ra[i], rb[i], p0, p1);
            fadd2(ra[i], rb[i], ra[i], rb[i], p2, p3);
            pk[i] = pack_e4m3x4(p0, p1, p2, p3);
          }
          st_shared_v4(p_row + ((c ^ (r_in & 7)) << 4), pk[0], pk[1], pk[2], pk[3]);
        }
        fence_proxy_async_smem();
        // Rescale O_X once it holds every earlier update (the update of
        // tile pc - 1 completes after all before it: one issuing thread,
        // MMAs in order); O_X += P_X(j) V_j waits for the arrival below.
        if (j > 0 && (unit_f != 1.f || __any_sync(0xffffffffu, resc))) {
          if (!__all_sync(0xffffffffu,
                          mbar_wait(o_done_bar(x, static_cast<int>((pc - 1) & 1)),
                                    ((pc - 1) >> 1) & 1, wc))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float f = alpha * unit_f;
#pragma unroll 1
          for (int c = 0; c < C::D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
            tmem_st32(tO + c * 32, o);
          }
        }
        tc_fence_before();
        mbar_arrive(p_full_bar(x, pb));
        // the row sum is not needed by the O update: after the arrival
        l_run += (((ra[0] + rb[0]) + (ra[1] + rb[1])) + ((ra[2] + rb[2]) + (ra[3] + rb[3]))) *
                 ex2(-lpw);
      }
      if (!ok) break;
      // ---------------- epilogue: O / l, lse ----------------
      if (!__all_sync(0xffffffffu, mbar_wait(&bar_o_final[x], tcount & 1, wc))) { ok = false; break; }
      tc_fence_after();
      const bool valid = row < ti.L;
      const float inv_l = (l_run > 0.f) ? 1.f / (r_unit * l_run) : 0.f;
      if (ti.part >= 0) {
        store_partial_row<C>(p, ti, x, r_in, tO, inv_l, m_run, l_run);
        tc_fence_before();
        mbar_arrive(&bar_o_free[x]);
        continue;
      }
      uint32_t *orow = nullptr;
      if (valid) {
        const size_t tok = static_cast<size_t>(ti.start) + row;
        orow = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(p.o) +
                                            (tok * p.H + ti.h) * p.d_out * 2);
      }
#pragma unroll 1
      for (int c = 0; c < p.d_out / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        if (valid) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
          uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            __stcs(dst + i, make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]));
        }
      }
      if (valid && p.lse != nullptr) {
        const float lse = (m_run + __log2f(l_run)) * 0.69314718055994531f;
        if constexpr (C::kVarlen)
          p.lse[static_cast<size_t>(ti.h) * p.T + ti.start + row] = lse;
        else
          p.lse[(static_cast<size_t>(ti.b) * p.H + ti.h) * p.N + row] = lse;
      }
      tc_fence_before();
      mbar_arrive(&bar_o_free[x]);
    }
  } else {
    // ------------------------------------------------------------------
    // 16-bit softmax warpgroups: x = 0 (sub-tile A) or 1 (sub-tile B), one
    // thread per query row
    // ------------------------------------------------------------------
    const int x = warp >> 2;
    const int wq = warp & 3;                 // TMEM lane quarter of this warp
    const int r_in = wq * 32 + lane;         // row within the sub-tile
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + x * C::kColS;
    const uint32_t tO = tmem + lane_base + C::kColO0 + x * C::D;
    // where P goes: over S, or (d = 64) its own columns
    const uint32_t tP = C::kSepP ? tmem + lane_base + C::kColP0 + x * 64 : tS;
    int s_cnt = 0, tcount = 0;
    unsigned pstore_cnt = 0;                 // kSepP: P tiles written so far
    bool ok = true;
    TileInfo ti;
    for (int t = blockIdx.x; ok && get_tile<C>(p, t, num_tiles, ti); t += gridDim.x, ++tcount) {
      const int nX = x == 0 ? ti.nA : ti.nB;
      const int row0 = ti.qt * 256 + x * 128;          // first row of the sub-tile
      const int row = row0 + r_in;                      // this thread's row
      float m_run = -INFINITY;                          // running max, log2 units
      float l_run = 0.f;
      for (int j = 0; j < nX; ++j) {
        if (!__all_sync(0xffffffffu, mbar_wait(&bar_s_full[x], s_cnt & 1, wc))) { ok = false; break; }
        ++s_cnt;
        tc_fence_after();
        uint32_t sv[128];
        float mx;                        // row maximum, from the load itself
        tmem_ld128_max(tS, sv, mx);      // the whole score row in one round trip
        if constexpr (C::kSepP) {        // S is in registers: the tensor core may overwrite it
          tc_fence_before();
          mbar_arrive(&bar_s_free[x]);
        }
        float cs = p.scale_log2;         // log2 units per raw score
        const int kbase = (ti.kb0 + j) * 128;
        if constexpr (C::kBias) {
          // scores to log2 units with the bias added: s * cs + bias * log2(e);
          // rows past the end read the last row's bias (their output is not
          // written), keys past the end are masked below
          constexpr float kLog2e = 1.4426950408889634f;
          const float *bp = p.bias + ti.b * p.bias_sb + ti.h * p.bias_sh +
                            static_cast<long long>(min(row, ti.L - 1)) * p.bias_sr + kbase;
          if (kbase + 128 <= ti.L) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              float4 bv[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) bv[u] = __ldg(reinterpret_cast<const float4 *>(bp + 32 * c) + u);
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const float bb[4] = {bv[u].x, bv[u].y, bv[u].z, bv[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int i = 32 * c + 4 * u + e;
                  sv[i] = __float_as_uint(fmaf(__uint_as_float(sv[i]), cs, bb[e] * kLog2e));
                }
              }
            }
          } else {
            const int nk = ti.L - kbase;
#pragma unroll
            for (int i = 0; i < 128; ++i)
              if (i < nk) sv[i] = __float_as_uint(fmaf(__uint_as_float(sv[i]), cs, __ldg(bp + i) * kLog2e));
          }
          cs = 1.f;
        }
        const bool need_mask = (kbase + 128 > ti.L) || (p.causal && kbase + 127 > row0);
        if (need_mask) {
          const int lim = p.causal ? min(ti.L, row + 1) : ti.L;   // keys < lim allowed
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (kbase + i >= lim) sv[i] = __float_as_uint(-INFINITY);
        }
        if (C::kBias || need_mask) {
          // the row changed after the load: its maximum from four independent
          // chains of three-input maxima
          float mq[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) mq[u] = __uint_as_float(sv[32 * u]);
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 1; i < 31; i += 2)
              mq[c] = fmax3(mq[c], __uint_as_float(sv[32 * c + i]), __uint_as_float(sv[32 * c + i + 1]));
#pragma unroll
          for (int c = 0; c < 4; ++c) mq[c] = fmaxf(mq[c], __uint_as_float(sv[32 * c + 31]));
          mx = fmax3(fmaxf(mq[0], mq[1]), mq[2], mq[3]);
        }
        const float m_tile = mx * cs;
        const float m_new = fmaxf(m_run, m_tile);
        const bool resc = m_new > m_run + C::kRescaleThresh;
        float alpha = 1.f;
        if (resc) {
          alpha = ex2(m_run - m_new);    // 0 when m_run = -inf
          l_run *= alpha;
          m_run = m_new;
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        if constexpr (C::kSepP) {
          // The previous O_X update must be complete before its P columns are
          // rewritten and before O_X is rescaled.
          if (pstore_cnt > 0 &&
              !__all_sync(0xffffffffu, mbar_wait(&bar_o_done[x], (pstore_cnt - 1) & 1, wc))) {
            ok = false;
            break;
          }
          ++pstore_cnt;
          tc_fence_after();
        }
        // x = s * cs - m in packed pairs; four independent packed row sums
        float ra[4] = {0.f, 0.f, 0.f, 0.f}, rb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            ffma2(x0, x1, __uint_as_float(sv[32 * c + 2 * i]), __uint_as_float(sv[32 * c + 2 * i + 1]),
                  cs, cs, -m_use, -m_use);
            const float p0 = ex2(x0), p1 = ex2(x1);
            fadd2(ra[i & 3], rb[i & 3], ra[i & 3], rb[i & 3], p0, p1);
            pk[i] = (C::E == Elem::BF16) ? pack_bf16(p0, p1) : pack_f16(p0, p1);
          }
          tmem_st16_nowait(tP + c * 16, pk);
        }
        tmem_wait_st();
        l_run += ((ra[0] + rb[0]) + (ra[1] + rb[1])) + ((ra[2] + rb[2]) + (ra[3] + rb[3]));
        // Rescale O after P is stored, when the score row is no longer live
        // (O_X may change until P_X(j) is published; PV_X(j) waits for that).
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
          for (int c = 0; c < C::D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + c * 32, o);
          }
        }
        tc_fence_before();
        mbar_arrive(&bar_p_full[x]);
      }
      if (!ok) break;
      // ---------------- epilogue: O / l, lse ----------------
      if (!__all_sync(0xffffffffu, mbar_wait(&bar_o_final[x], tcount & 1, wc))) { ok = false; break; }
      tc_fence_after();
      const bool valid = row < ti.L;
      const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
      if (ti.part >= 0) {
        store_partial_row<C>(p, ti, x, r_in, tO, inv_l, m_run, l_run);
        tc_fence_before();
        mbar_arrive(&bar_o_free[x]);
        continue;
      }
      uint32_t *orow = nullptr;
      if (valid) {
        const size_t tok = static_cast<size_t>(ti.start) + row;
        orow = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(p.o) +
                                            ((tok * p.H + ti.h) * C::D) * 2);
      }
#pragma unroll
      for (int c = 0; c < C::D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        if (valid) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a = __uint_as_float(o[2 * i]) * inv_l;
            const float b = __uint_as_float(o[2 * i + 1]) * inv_l;
            w[i] = (C::E == Elem::F16) ? pack_f16(a, b) : pack_bf16(a, b);
          }
          uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            __stcs(dst + i, make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]));
        }
      }
      if (valid && p.lse != nullptr) {
        const float lse = (m_run + __log2f(l_run)) * 0.69314718055994531f;
        if constexpr (C::kVarlen)
          p.lse[static_cast<size_t>(ti.h) * p.T + ti.start + row] = lse;
        else
          p.lse[(static_cast<size_t>(ti.b) * p.H + ti.h) * p.N + row] = lse;
      }
      tc_fence_before();
      mbar_arrive(&bar_o_free[x]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace attn
