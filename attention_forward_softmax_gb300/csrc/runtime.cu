// runtime.cu -- host side of the C ABI: argument validation, per-device
// workspace and status word, tensor-map encoding, the varlen tile-list
// builder, and the attn_fwd / attn_fwd_varlen / attn_fwd_fp8 entry points.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "internal.h"

namespace attn {

namespace {
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn g_encode = nullptr;
}  // namespace

long long wait_budget() {
  static long long b = [] {
    const char *e = std::getenv("ATTN_WAIT_BUDGET_CYCLES");
    long long v = e ? std::atoll(e) : 0;
    return v > 0 ? v : (1LL << 31);   // about one second at 2 GHz
  }();
  return b;
}

attn_status_t device_state(DeviceState **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState &ds = g_dev[dev];
  if (ds.status == nullptr) {
    if (cudaDeviceGetAttribute(&ds.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    void *p = nullptr;
    if (cudaMalloc(&p, 256) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemset(p, 0, 256) != cudaSuccess) return ATTN_ERR_CUDA;
    ds.status = static_cast<int *>(p);
    ds.num_entries = ds.status + 1;
    ds.scratch_amax = reinterpret_cast<float *>(ds.status + 4);
  }
  *out = &ds;
  return ATTN_OK;
}

attn_status_t ensure_tiles(DeviceState *ds, size_t entries) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (ds->tiles_cap >= entries) return ATTN_OK;
  size_t cap = ds->tiles_cap ? ds->tiles_cap : 4096;
  while (cap < entries) cap *= 2;
  if (ds->tiles) {
    // The old list may still be read by queued work: wait before freeing.
    if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
    cudaFree(ds->tiles);
    ds->tiles = nullptr;
    ds->tiles_cap = 0;
  }
  void *p = nullptr;
  if (cudaMalloc(&p, cap * sizeof(int2)) != cudaSuccess) return ATTN_ERR_CUDA;
  ds->tiles = static_cast<int2 *>(p);
  ds->tiles_cap = cap;
  return ATTN_OK;
}

namespace {
// Grows a cached device buffer to at least `bytes`; the old one may still be
// used by queued work, so the device is synchronised before it is freed.
attn_status_t grow_workspace(float **buf, size_t *cap_bytes, size_t bytes) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (*cap_bytes >= bytes) return ATTN_OK;
  size_t cap = *cap_bytes ? *cap_bytes : (1u << 20);
  while (cap < bytes) cap *= 2;
  if (*buf) {
    if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
    cudaFree(*buf);
    *buf = nullptr;
    *cap_bytes = 0;
  }
  void *p = nullptr;
  if (cudaMalloc(&p, cap) != cudaSuccess) return ATTN_ERR_CUDA;
  *buf = static_cast<float *>(p);
  *cap_bytes = cap;
  return ATTN_OK;
}
}  // namespace

attn_status_t ensure_split_workspace(DeviceState *ds, size_t bytes) {
  return grow_workspace(&ds->split_ws, &ds->split_ws_bytes, bytes);
}

attn_status_t ensure_bwd_workspace(DeviceState *ds, size_t bytes) {
  return grow_workspace(&ds->bwd_ws, &ds->bwd_ws_bytes, bytes);
}

attn_status_t plan_tail_split(DeviceState *ds, LaunchArgs &a) {
  a.split_rem = 0;
  if (a.causal || a.num_tiles <= 0 || ds->num_sms <= 0) return ATTN_OK;
  if (a.dq != nullptr && a.d != 128) return ATTN_OK;   // e4m3 at d = 64: partials are 128 wide
  const int grid = a.num_tiles < ds->num_sms ? a.num_tiles : ds->num_sms;
  const int rem = a.num_tiles % grid;
  // worth it only when the last wave is at most half full, and each half
  // gets at least one key tile
  if (rem == 0 || 2 * rem > grid || (a.N + 127) / 128 < 2) return ATTN_OK;
  const size_t rows = static_cast<size_t>(rem) * 2 * 256;
  attn_status_t st = grow_workspace(&ds->fwd_split_ws, &ds->fwd_split_ws_bytes,
                                    rows * (a.d + 1) * sizeof(float));
  if (st != ATTN_OK) return st;
  a.split_rem = rem;
  a.part_o = ds->fwd_split_ws;
  a.part_lse = ds->fwd_split_ws + rows * a.d;
  return ATTN_OK;
}

attn_status_t encode_tiled(CUtensorMap *map, CUtensorMapDataType dtype, int rank, const void *ptr,
                           const cuuint64_t *dims, const cuuint64_t *strides,
                           const cuuint32_t *box, CUtensorMapSwizzle swizzle) {
  if (g_encode == nullptr) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode == nullptr) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return ATTN_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeFn>(fn);
    }
  }
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void *>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_INVALID_ARG;
}

// ---------------------------------------------------------------------------
// Varlen schedule: validate cu_seqlens and list the (sequence, query-tile)
// work tiles heaviest first (counting sort on the number of key tiles the
// tile's heavier sub-tile scores).  One CTA; the list length goes to
// *num_entries (0 when cu_seqlens is malformed, which is also reported in
// the status word).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int tile_work(int L, int qt, int causal) {
  const int nkv = (L + 127) / 128;
  if (!causal) return nkv;
  return (qt * 256 + 128 < L) ? min(2 * qt + 2, nkv) : min(2 * qt + 1, nkv);
}

constexpr int kSchedThreads = 1024;
constexpr int kMaxWorkKey = 4096;

__global__ void __launch_bounds__(kSchedThreads)
    varlen_schedule_kernel(const int *cu, int nseq, int T, int max_seqlen, int causal, int2 *tiles,
                           int capacity, int *num_entries, int *status) {
  __shared__ int hist[kMaxWorkKey];
  __shared__ int bad;
  const int nkeys = min(kMaxWorkKey, (max_seqlen + 127) / 128 + 1);
  if (threadIdx.x == 0) bad = 0;
  for (int i = threadIdx.x; i < nkeys; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int s = threadIdx.x; s < nseq; s += blockDim.x) {
    const int a = cu[s], b = cu[s + 1];
    if ((s == 0 && a != 0) || b < a || b - a > max_seqlen || (s == nseq - 1 && b != T)) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) {
      *num_entries = 0;
      atomicCAS(status, 0, 6 /* ATTN_ERR_BAD_SEQLENS */);
    }
    return;
  }
  for (int s = threadIdx.x; s < nseq; s += blockDim.x) {
    const int L = cu[s + 1] - cu[s];
    for (int qt = 0; qt * 256 < L; ++qt) atomicAdd(&hist[min(tile_work(L, qt, causal), nkeys - 1)], 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {   // exclusive offsets, heaviest key first
    int run = 0;
    for (int k = nkeys - 1; k >= 0; --k) {
      const int c = hist[k];
      hist[k] = run;
      run += c;
    }
    *num_entries = min(run, capacity);
  }
  __syncthreads();
  for (int s = threadIdx.x; s < nseq; s += blockDim.x) {
    const int L = cu[s + 1] - cu[s];
    for (int qt = 0; qt * 256 < L; ++qt) {
      const int pos = atomicAdd(&hist[min(tile_work(L, qt, causal), nkeys - 1)], 1);
      if (pos < capacity) tiles[pos] = make_int2(s, qt);
    }
  }
}

cudaError_t launch_varlen_schedule(const int *cu_seqlens, int nseq, int total_tokens,
                                   int max_seqlen, int causal, int2 *tiles, int capacity,
                                   int *num_entries, int *status, cudaStream_t s) {
  varlen_schedule_kernel<<<1, kSchedThreads, 0, s>>>(cu_seqlens, nseq, total_tokens, max_seqlen,
                                                     causal ? 1 : 0, tiles, capacity, num_entries,
                                                     status);
  return cudaGetLastError();
}

namespace {

attn_status_t check_common(const void *q, const void *k, const void *v, const void *o,
                           const float *lse, int H, int d, float scale) {
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (H < 1 || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_MISALIGNED;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_MISALIGNED;
  return ATTN_OK;
}

// A piece of the work of a host-buffer forward: heads h0 .. h0 + nh - 1 of
// batch entry b.
struct HostChunk {
  int b, h0, nh;
};

// Host-buffer pipeline of attn_fwd_host and attn_fwd_fp8_host.  The work is
// cut into chunks: whole batch entries, except that the first and the last
// entry are cut into groups of hg heads -- the fewest heads whose 256-row
// tiles still fill every SM once -- so the compute starts after a smaller
// first copy and little is left after the last one.  A chunk's rows are
// strided in the host arrays (nh of H heads per token): 2-D copies move
// them to and from compact staging buffers.  Per chunk, on kHostSets
// staging sets in turn: q, k, v copied in on the copy-in stream (once the
// set's previous chunk has been computed); `compute` queued on the caller's
// stream or the second compute stream in turn (one chunk's last wave
// overlaps the next chunk's first), once the inputs are in and the set's
// previous outputs have left; o and lse copied out on the copy-out stream.
// A set holds q, k, v, o, lse of up to one batch entry and `extra_bytes`
// more for `compute`; `pre_bytes` from `pre_src` (host) go once to a
// device area after the sets, before the first chunk.
template <class Compute>
attn_status_t host_pipeline(DeviceState *ds, const void *q, const void *k, const void *v, void *o,
                            float *lse, int B, int H, int N, int d, size_t extra_bytes,
                            const void *pre_src, size_t pre_bytes, cudaStream_t s,
                            Compute compute) {
  constexpr int S = DeviceState::kHostSets;
  const size_t row = static_cast<size_t>(H) * d * 2;            // one token of q, k, v or o
  const size_t per_b = static_cast<size_t>(N) * row;            // one batch entry
  const size_t lse_b = static_cast<size_t>(H) * N * sizeof(float);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t set_bytes = 4 * up(per_b) + up(lse_b) + up(extra_bytes);
  attn_status_t st = grow_workspace(&ds->host_ws, &ds->host_ws_bytes, S * set_bytes + up(pre_bytes));
  if (st != ATTN_OK) return st;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (ds->h2d == nullptr) {
      if (cudaStreamCreateWithFlags(&ds->h2d, cudaStreamNonBlocking) != cudaSuccess ||
          cudaStreamCreateWithFlags(&ds->d2h, cudaStreamNonBlocking) != cudaSuccess ||
          cudaStreamCreateWithFlags(&ds->comp2, cudaStreamNonBlocking) != cudaSuccess ||
          cudaEventCreateWithFlags(&ds->ev_start, cudaEventDisableTiming) != cudaSuccess)
        return ATTN_ERR_CUDA;
      for (int i = 0; i < S; ++i)
        if (cudaEventCreateWithFlags(&ds->ev_in[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&ds->ev_comp[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&ds->ev_out[i], cudaEventDisableTiming) != cudaSuccess)
          return ATTN_ERR_CUDA;
    }
  }
  const int nqt = (N + 255) / 256;
  int hg = H;
  for (int x = 1; x < H; ++x)
    if (H % x == 0 && static_cast<long long>(x) * nqt >= ds->num_sms) {
      hg = x;
      break;
    }
  std::vector<HostChunk> chunks;
  for (int b = 0; b < B; ++b) {
    if ((b == 0 || b == B - 1) && hg < H)
      for (int h0 = 0; h0 < H; h0 += hg) chunks.push_back({b, h0, hg});
    else
      chunks.push_back({b, 0, H});
  }
  const char *qh = static_cast<const char *>(q), *kh = static_cast<const char *>(k);
  const char *vh = static_cast<const char *>(v);
  char *oh = static_cast<char *>(o);
  char *ws = reinterpret_cast<char *>(ds->host_ws);
  char *pre = ws + S * set_bytes;
  bool ok = true;
  auto chk = [&ok](cudaError_t e) { ok = ok && e == cudaSuccess; };
  // everything queued on the caller's stream before this call comes first
  chk(cudaEventRecord(ds->ev_start, s));
  chk(cudaStreamWaitEvent(ds->h2d, ds->ev_start, 0));
  if (pre_bytes > 0) chk(cudaMemcpyAsync(pre, pre_src, pre_bytes, cudaMemcpyHostToDevice, ds->h2d));
  const int nc = static_cast<int>(chunks.size());
  int last_set = 0;
  for (int c = 0; ok && c < nc; ++c) {
    const HostChunk ch = chunks[c];
    const int set = c % S;
    last_set = set;
    char *dq = ws + set * set_bytes, *dk = dq + up(per_b), *dv = dk + up(per_b);
    char *dout = dv + up(per_b);
    float *dlse = reinterpret_cast<float *>(dout + up(per_b));
    char *extra = dout + up(per_b) + up(lse_b);
    const size_t w = static_cast<size_t>(ch.nh) * d * 2;        // bytes of a chunk row
    const size_t hoff = static_cast<size_t>(ch.b) * per_b + static_cast<size_t>(ch.h0) * d * 2;
    // inputs, once chunk c - S (same set) has been computed (one copy
    // stream: a second one measured slower, the two share the host link)
    if (c >= S) chk(cudaStreamWaitEvent(ds->h2d, ds->ev_comp[set], 0));
    chk(cudaMemcpy2DAsync(dq, w, qh + hoff, row, w, N, cudaMemcpyHostToDevice, ds->h2d));
    chk(cudaMemcpy2DAsync(dk, w, kh + hoff, row, w, N, cudaMemcpyHostToDevice, ds->h2d));
    chk(cudaMemcpy2DAsync(dv, w, vh + hoff, row, w, N, cudaMemcpyHostToDevice, ds->h2d));
    chk(cudaEventRecord(ds->ev_in[set], ds->h2d));
    cudaStream_t cs = (c & 1) ? ds->comp2 : s;
    chk(cudaStreamWaitEvent(cs, ds->ev_in[set], 0));
    if (c >= S) chk(cudaStreamWaitEvent(cs, ds->ev_out[set], 0));
    if (!ok) break;
    if ((st = compute(ch, dq, dk, dv, dout, lse ? dlse : nullptr, extra, pre, cs)) != ATTN_OK)
      return st;
    chk(cudaEventRecord(ds->ev_comp[set], cs));
    // outputs of the chunk
    chk(cudaStreamWaitEvent(ds->d2h, ds->ev_comp[set], 0));
    chk(cudaMemcpy2DAsync(oh + hoff, row, dout, w, w, N, cudaMemcpyDeviceToHost, ds->d2h));
    if (lse)
      chk(cudaMemcpyAsync(lse + (static_cast<size_t>(ch.b) * H + ch.h0) * N, dlse,
                          static_cast<size_t>(ch.nh) * N * sizeof(float), cudaMemcpyDeviceToHost,
                          ds->d2h));
    chk(cudaEventRecord(ds->ev_out[set], ds->d2h));
  }
  // later work on the caller's stream sees the outputs (the copy-out stream
  // runs in order and every copy-out follows its chunk's compute, so its
  // last event covers both compute streams)
  if (ok) chk(cudaStreamWaitEvent(s, ds->ev_out[last_set], 0));
  return ok ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

// The dense 16-bit forward; allow_split = false keeps the last wave whole
// (no use of the per-device split workspace, so two such launches may run
// at once on different streams).
static attn_status_t fwd_dense(const void *q, const void *k, const void *v, void *o, float *lse,
                               int B, int H, int H_kv, int N, int d, float scale, int causal,
                               attn_dtype_t dtype, bool allow_split, cudaStream_t s) {
  attn_status_t st = check_common(q, k, v, o, lse, H, d, scale);
  if (st != ATTN_OK) return st;
  if (B < 1 || N < 1 || H_kv < 1 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  const long long tokens = static_cast<long long>(B) * N;
  const long long tiles = static_cast<long long>(B) * H * ((N + 255) / 256);
  if (tokens * H * d > (1LL << 40) || tiles > (1LL << 30)) return ATTN_ERR_TOO_LARGE;
  DeviceState *ds = nullptr;
  if ((st = device_state(&ds)) != ATTN_OK) return st;
  LaunchArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.B = B; a.H = H; a.Hkv = H_kv; a.N = N; a.d = d;
  a.T = static_cast<int>(tokens > 0x7fffffff ? 0 : tokens);
  a.scale = scale; a.causal = causal ? 1 : 0;
  a.num_tiles = static_cast<int>(tiles);
  a.status = ds->status; a.budget = wait_budget(); a.num_sms = ds->num_sms;
  if (allow_split && (st = plan_tail_split(ds, a)) != ATTN_OK) return st;
  return dtype == ATTN_BF16 ? launch_attn_bf16(a, false, s) : launch_attn_f16(a, false, s);
}

attn_status_t attn_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse,
                           int B, int H, int H_kv, int N, int d, float scale, int causal,
                           attn_dtype_t dtype, void *stream) {
  return fwd_dense(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, dtype, true,
                   static_cast<cudaStream_t>(stream));
}

attn_status_t attn_fwd_bias(const void *q, const void *k, const void *v, const float *bias,
                            long long bias_stride_b, long long bias_stride_h,
                            long long bias_stride_row, void *o, float *lse, int B, int H,
                            int H_kv, int N, int d, float scale, int causal, attn_dtype_t dtype,
                            void *stream) {
  attn_status_t st = check_common(q, k, v, o, lse, H, d, scale);
  if (st != ATTN_OK) return st;
  if (!bias || B < 1 || N < 1 || H_kv < 1 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (bias_stride_b < 0 || bias_stride_h < 0 || bias_stride_row < 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  // every bias row starts on a 16-byte boundary (vector loads)
  if (!aligned16(bias) || (bias_stride_b & 3) || (bias_stride_h & 3) || (bias_stride_row & 3))
    return ATTN_ERR_MISALIGNED;
  const long long tokens = static_cast<long long>(B) * N;
  const long long tiles = static_cast<long long>(B) * H * ((N + 255) / 256);
  if (tokens * H * d > (1LL << 40) || tiles > (1LL << 30)) return ATTN_ERR_TOO_LARGE;
  DeviceState *ds = nullptr;
  if ((st = device_state(&ds)) != ATTN_OK) return st;
  LaunchArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.B = B; a.H = H; a.Hkv = H_kv; a.N = N; a.d = d;
  a.T = static_cast<int>(tokens > 0x7fffffff ? 0 : tokens);
  a.scale = scale; a.causal = causal ? 1 : 0;
  a.num_tiles = static_cast<int>(tiles);
  a.bias = bias; a.bias_sb = bias_stride_b; a.bias_sh = bias_stride_h;
  a.bias_sr = bias_stride_row;
  a.status = ds->status; a.budget = wait_budget(); a.num_sms = ds->num_sms;
  if ((st = plan_tail_split(ds, a)) != ATTN_OK) return st;
  return launch_attn_bias(a, dtype == ATTN_BF16, static_cast<cudaStream_t>(stream));
}

attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                       int H, int N, int d, float scale, int causal, attn_dtype_t dtype,
                       void *stream) {
  return attn_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, scale, causal, dtype, stream);
}

attn_status_t attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int H, int N, int d, float scale, int causal,
                            attn_dtype_t dtype, void *stream) {
  attn_status_t st = check_common(q, k, v, o, lse, H, d, scale);
  if (st != ATTN_OK) return st;
  if (B < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(N) * H * d > (1LL << 40) / B) return ATTN_ERR_TOO_LARGE;
  DeviceState *ds = nullptr;
  if ((st = device_state(&ds)) != ATTN_OK) return st;
  // each chunk: the dense forward on its compact buffers, the last wave
  // whole (two chunks may run at once; the split workspace is shared)
  auto compute = [&](const HostChunk &ch, char *dq, char *dk, char *dv, char *dout, float *dlse,
                     char *, char *, cudaStream_t cs) {
    return fwd_dense(dq, dk, dv, dout, dlse, 1, ch.nh, ch.nh, N, d, scale, causal, dtype, false,
                     cs);
  };
  return host_pipeline(ds, q, k, v, o, lse, B, H, N, d, 0, nullptr, 0,
                       static_cast<cudaStream_t>(stream), compute);
}

attn_status_t attn_fwd_varlen_gqa(const void *q, const void *k, const void *v, void *o,
                                  float *lse, const int32_t *cu_seqlens, int nseq,
                                  int total_tokens, int max_seqlen, int H, int H_kv, int d,
                                  float scale, int causal, attn_dtype_t dtype, void *stream) {
  attn_status_t st = check_common(q, k, v, o, lse, H, d, scale);
  if (st != ATTN_OK) return st;
  if (!cu_seqlens || nseq < 1 || total_tokens < 1 || max_seqlen < 1) return ATTN_ERR_INVALID_ARG;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return ATTN_ERR_MISALIGNED;
  const long long entries = static_cast<long long>(total_tokens) / 256 + nseq;
  if (static_cast<long long>(total_tokens) * H * d > (1LL << 40) || entries * H > (1LL << 30))
    return ATTN_ERR_TOO_LARGE;
  DeviceState *ds = nullptr;
  if ((st = device_state(&ds)) != ATTN_OK) return st;
  if ((st = ensure_tiles(ds, static_cast<size_t>(entries))) != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  varlen_schedule_kernel<<<1, kSchedThreads, 0, s>>>(cu_seqlens, nseq, total_tokens, max_seqlen,
                                                     causal ? 1 : 0, ds->tiles,
                                                     static_cast<int>(entries), ds->num_entries,
                                                     ds->status);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  LaunchArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.B = nseq; a.H = H; a.Hkv = H_kv; a.N = max_seqlen; a.d = d; a.T = total_tokens;
  a.scale = scale; a.causal = causal ? 1 : 0;
  a.cu_seqlens = cu_seqlens; a.tiles = ds->tiles; a.num_entries = ds->num_entries;
  a.num_tiles = static_cast<int>(entries * H);
  a.status = ds->status; a.budget = wait_budget(); a.num_sms = ds->num_sms;
  return dtype == ATTN_BF16 ? launch_attn_bf16(a, true, s) : launch_attn_f16(a, true, s);
}

attn_status_t attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                              const int32_t *cu_seqlens, int nseq, int total_tokens,
                              int max_seqlen, int H, int d, float scale, int causal,
                              attn_dtype_t dtype, void *stream) {
  return attn_fwd_varlen_gqa(q, k, v, o, lse, cu_seqlens, nseq, total_tokens, max_seqlen, H, H,
                             d, scale, causal, dtype, stream);
}

// The e4m3 forward; allow_split as for fwd_dense.
static attn_status_t fwd_fp8(const void *q8, const void *k8, const void *v8,
                             const float *descale_q, const float *descale_k,
                             const float *descale_v, void *o, float *lse, int B, int H, int N,
                             int d, float scale, int causal, bool allow_split, cudaStream_t s) {
  attn_status_t st = check_common(q8, k8, v8, o, lse, H, d, scale);
  if (st != ATTN_OK) return st;
  if (B < 1 || N < 1 || !descale_q || !descale_k || !descale_v) return ATTN_ERR_INVALID_ARG;
  if (d != 128 && d != 64) return ATTN_ERR_UNSUPPORTED;
  const long long tokens = static_cast<long long>(B) * N;
  const long long tiles = static_cast<long long>(B) * H * ((N + 255) / 256);
  if (tokens * H * d > (1LL << 40) || tiles > (1LL << 30)) return ATTN_ERR_TOO_LARGE;
  DeviceState *ds = nullptr;
  if ((st = device_state(&ds)) != ATTN_OK) return st;
  LaunchArgs a{};
  a.q = q8; a.k = k8; a.v = v8; a.o = o; a.lse = lse;
  a.B = B; a.H = H; a.Hkv = H; a.N = N; a.d = d;
  a.T = static_cast<int>(tokens > 0x7fffffff ? 0 : tokens);
  a.scale = scale; a.causal = causal ? 1 : 0;
  a.num_tiles = static_cast<int>(tiles);
  a.dq = descale_q; a.dk = descale_k; a.dv = descale_v;
  a.status = ds->status; a.budget = wait_budget(); a.num_sms = ds->num_sms;
  if (allow_split && (st = plan_tail_split(ds, a)) != ATTN_OK) return st;
  return launch_attn_e4m3(a, s);
}

attn_status_t attn_fwd_fp8(const void *q8, const void *k8, const void *v8, const float *descale_q,
                           const float *descale_k, const float *descale_v, void *o, float *lse,
                           int B, int H, int N, int d, float scale, int causal, void *stream) {
  return fwd_fp8(q8, k8, v8, descale_q, descale_k, descale_v, o, lse, B, H, N, d, scale, causal,
                 true, static_cast<cudaStream_t>(stream));
}

attn_status_t attn_fwd_fp8_host(const void *q, const void *k, const void *v, const int8_t *signs,
                                void *o, float *lse, int B, int H, int N, int d, float scale,
                                int causal, void *stream) {
  attn_status_t st = check_common(q, k, v, o, lse, H, d, scale);
  if (st != ATTN_OK) return st;
  if (B < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(N) * H * d > (1LL << 40) / B) return ATTN_ERR_TOO_LARGE;
  DeviceState *ds = nullptr;
  if ((st = device_state(&ds)) != ATTN_OK) return st;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const int nblk = (N + 127) / 128;
  const size_t code_b = up(static_cast<size_t>(N) * H * d);             // e4m3 codes of one entry
  const size_t dsc_b = up(static_cast<size_t>(H) * nblk * sizeof(float));
  // each chunk: block quantisation (with the rotation when signs are given)
  // of its compact q, k, v, then the e4m3 forward, the last wave whole
  auto compute = [&](const HostChunk &ch, char *dq, char *dk, char *dv, char *dout, float *dlse,
                     char *extra, char *pre, cudaStream_t cs) {
    char *q8 = extra, *k8 = q8 + code_b, *v8 = k8 + code_b;
    float *dsq = reinterpret_cast<float *>(v8 + code_b);
    float *dsk = reinterpret_cast<float *>(reinterpret_cast<char *>(dsq) + dsc_b);
    float *dsv = reinterpret_cast<float *>(reinterpret_cast<char *>(dsk) + dsc_b);
    attn_status_t r = qkv_block_quant_hadamard(dq, dk, dv, q8, k8, v8, dsq, dsk, dsv,
                                               signs ? reinterpret_cast<const int8_t *>(pre)
                                                     : nullptr,
                                               0, 1, ch.nh, N, d, cs);
    if (r != ATTN_OK) return r;
    return fwd_fp8(q8, k8, v8, dsq, dsk, dsv, dout, dlse, 1, ch.nh, N, d, scale, causal, false,
                   cs);
  };
  return host_pipeline(ds, q, k, v, o, lse, B, H, N, d, 3 * code_b + 3 * dsc_b, signs,
                       signs ? static_cast<size_t>(d) : 0, static_cast<cudaStream_t>(stream),
                       compute);
}

attn_status_t attn_get_status(void *stream) {
  DeviceState *ds = nullptr;
  attn_status_t st = device_state(&ds);
  if (st != ATTN_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, ds->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (h != 0 && cudaMemset(ds->status, 0, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  return static_cast<attn_status_t>(h);
}

const char *attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported head dimension or dtype";
    case ATTN_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
    case ATTN_ERR_LAUNCH: return "kernel launch failed";
    case ATTN_ERR_TIMEOUT: return "device pipeline wait timed out";
    case ATTN_ERR_BAD_SEQLENS: return "malformed cu_seqlens";
    case ATTN_ERR_CUDA: return "CUDA runtime error";
    case ATTN_ERR_TOO_LARGE: return "problem size exceeds the supported index range";
  }
  return "unknown status";
}

void attn_shutdown(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (int d = 0; d < kMaxDevices; ++d) {
    DeviceState &ds = g_dev[d];
    if (ds.status == nullptr && ds.tiles == nullptr && ds.split_ws == nullptr &&
        ds.bwd_ws == nullptr && ds.fwd_split_ws == nullptr && ds.host_ws == nullptr)
      continue;
    if (cudaSetDevice(d) != cudaSuccess) continue;
    cudaDeviceSynchronize();
    if (ds.tiles) cudaFree(ds.tiles);
    if (ds.split_ws) cudaFree(ds.split_ws);
    if (ds.bwd_ws) cudaFree(ds.bwd_ws);
    if (ds.fwd_split_ws) cudaFree(ds.fwd_split_ws);
    if (ds.host_ws) cudaFree(ds.host_ws);
    for (int i = 0; i < DeviceState::kHostSets; ++i) {
      if (ds.ev_in[i]) cudaEventDestroy(ds.ev_in[i]);
      if (ds.ev_comp[i]) cudaEventDestroy(ds.ev_comp[i]);
      if (ds.ev_out[i]) cudaEventDestroy(ds.ev_out[i]);
    }
    if (ds.ev_start) cudaEventDestroy(ds.ev_start);
    if (ds.h2d) cudaStreamDestroy(ds.h2d);
    if (ds.d2h) cudaStreamDestroy(ds.d2h);
    if (ds.comp2) cudaStreamDestroy(ds.comp2);
    if (ds.status) cudaFree(ds.status);
    ds = DeviceState{};
  }
  cudaSetDevice(cur);
}

uint32_t attn_version(void) { return 0x00000100u; }

}  // extern "C"
