// noalloc.cu -- attn_fwd_varlen_noalloc: the packed variable-length attention
// forward pass for callers that cannot allocate device memory.
//
// Who needs it: code whose device memory is planned by someone else -- a
// plugin or custom op inside a framework or inference runtime that hands it
// only its inputs, outputs and nothing else, or a service that forbids
// allocation after start-up.  For them the regular attn_fwd_varlen is
// unusable: on first use, and whenever a larger tile list is needed, it
// calls cudaMalloc (and cudaFree, which waits for the whole device).
//
// This variant keeps its scratch -- the device status word, the tile-list
// length and the tile list itself -- in one file-scope __device__ array of
// fixed size, which exists on every GPU that loads the library until the
// process exits.  It calls no cudaMalloc, cudaFree or allocating library
// routine.  Limits and sharing rules are stated beside the declaration in
// attn.h.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"

namespace attn {
namespace {

// Scratch layout: [0, 4) status word, [4, 8) tile-list length, [256, ...)
// tile list of (sequence, query tile) pairs.
constexpr int kNoAllocMaxEntries = 32768;
constexpr size_t kNoAllocHeader = 256;
constexpr size_t kNoAllocBytes = kNoAllocHeader + kNoAllocMaxEntries * sizeof(int2);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

unsigned char *g_scratch_ptr[kMaxDevices] = {};   // device address of g_noalloc_scratch, per device
int g_num_sms[kMaxDevices] = {};
std::mutex g_setup_mu;

// Once per device, with that device current: look up the device address of
// the scratch array (the host-side name is only a stand-in for it) and the
// SM count.  Neither allocates.
attn_status_t setup(int dev, unsigned char **scratch, int *num_sms) {
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return ATTN_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    g_num_sms[dev] = sms;
    g_scratch_ptr[dev] = static_cast<unsigned char *>(ptr);
  }
  *scratch = g_scratch_ptr[dev];
  *num_sms = g_num_sms[dev];
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" attn_status_t attn_fwd_varlen_noalloc(const void *q, const void *k, const void *v,
                                                 void *o, float *lse, const int32_t *cu_seqlens,
                                                 int nseq, int total_tokens, int max_seqlen,
                                                 int H, int d, float scale, int causal,
                                                 attn_dtype_t dtype, int32_t *status,
                                                 void *stream) {
  if (!q || !k || !v || !o || !cu_seqlens) return ATTN_ERR_INVALID_ARG;
  if (H < 1 || nseq < 1 || total_tokens < 1 || max_seqlen < 1 || !std::isfinite(scale))
    return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_MISALIGNED;
  if ((lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) ||
      (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) ||
      (status && (reinterpret_cast<uintptr_t>(status) & 3u)))
    return ATTN_ERR_MISALIGNED;
  // Every sequence contributes at most L/256 + 1 work tiles.
  const long long entries = static_cast<long long>(total_tokens) / 256 + nseq;
  if (entries > kNoAllocMaxEntries) return ATTN_ERR_TOO_LARGE;
  if (static_cast<long long>(total_tokens) * H * d > (1LL << 40) || entries * H > (1LL << 30))
    return ATTN_ERR_TOO_LARGE;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  unsigned char *scratch = nullptr;
  int num_sms = 0;
  attn_status_t st = setup(dev, &scratch, &num_sms);
  if (st != ATTN_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int *dev_status = status ? reinterpret_cast<int *>(status) : reinterpret_cast<int *>(scratch);
  int *num_entries = reinterpret_cast<int *>(scratch + 4);
  int2 *tiles = reinterpret_cast<int2 *>(scratch + kNoAllocHeader);
  // The scratch keeps the previous call's contents.  The status word must
  // start at zero (kernels only ever replace a zero with an error code);
  // the tile list and its length are rewritten in full by the builder.
  if (cudaMemsetAsync(dev_status, 0, sizeof(int), s) != cudaSuccess) return ATTN_ERR_CUDA;
  if (launch_varlen_schedule(cu_seqlens, nseq, total_tokens, max_seqlen, causal ? 1 : 0, tiles,
                             static_cast<int>(entries), num_entries, dev_status, s) != cudaSuccess)
    return ATTN_ERR_LAUNCH;

  LaunchArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.B = nseq; a.H = H; a.Hkv = H; a.N = max_seqlen; a.d = d; a.T = total_tokens;
  a.scale = scale; a.causal = causal ? 1 : 0;
  a.cu_seqlens = cu_seqlens; a.tiles = tiles; a.num_entries = num_entries;
  a.num_tiles = static_cast<int>(entries * H);
  a.status = dev_status; a.budget = wait_budget(); a.num_sms = num_sms;
  return dtype == ATTN_BF16 ? launch_attn_bf16(a, true, s) : launch_attn_f16(a, true, s);
}
