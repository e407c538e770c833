// internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn.h"

namespace attn {

// Devices the per-device host state is kept for (device ordinals 0 .. 63).
constexpr int kMaxDevices = 64;

// Everything one attention launch needs (already validated).
struct LaunchArgs {
  const void *q, *k, *v;
  void *o;
  float *lse;
  int B, H, N, d, T;
  int Hkv;                   // K/V heads (H_kv divides H)
  float scale;
  int causal;
  const int *cu_seqlens;     // varlen
  const int2 *tiles;         // varlen tile list (device)
  const int *num_entries;    // varlen tile-list length (device)
  int num_tiles;             // dense: exact; varlen: upper bound (x H)
  const float *dq, *dk, *dv; // e4m3 descales
  const float *bias;         // additive score bias (or null)
  long long bias_sb, bias_sh, bias_sr;
  int *status;
  long long budget;
  int num_sms;
  // dense, non-causal: the last split_rem tiles run as two key halves each
  // (work items num_tiles - split_rem on; num_tiles counts tiles), their
  // partials in part_o / part_lse; split_rem = 0: no split
  int split_rem;
  float *part_o, *part_lse;
};

attn_status_t launch_attn_bf16(const LaunchArgs &a, bool varlen, cudaStream_t s);
attn_status_t launch_attn_f16(const LaunchArgs &a, bool varlen, cudaStream_t s);
attn_status_t launch_attn_e4m3(const LaunchArgs &a, cudaStream_t s);
attn_status_t launch_attn_bias(const LaunchArgs &a, bool bf16, cudaStream_t s);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).  dims/strides/box are innermost-first; strides has
// rank-1 entries in bytes.
attn_status_t encode_tiled(CUtensorMap *map, CUtensorMapDataType dtype, int rank, const void *ptr,
                           const cuuint64_t *dims, const cuuint64_t *strides,
                           const cuuint32_t *box, CUtensorMapSwizzle swizzle);

// Per-device state.
struct DeviceState {
  int *status = nullptr;        // device status word
  int *num_entries = nullptr;   // varlen tile-list length
  float *scratch_amax = nullptr;  // per-tensor quantisation: 3 floats
  int2 *tiles = nullptr;        // varlen tile list
  size_t tiles_cap = 0;
  float *split_ws = nullptr;    // paged decoding: per-split partial O and lse
  size_t split_ws_bytes = 0;
  float *bwd_ws = nullptr;      // backward: fp32 dQ accumulator and rowsum(dO * O)
  size_t bwd_ws_bytes = 0;
  float *fwd_split_ws = nullptr;  // forward: partials of the split last tiles
  size_t fwd_split_ws_bytes = 0;
  // host-buffer forward (attn_fwd_host): kHostSets device staging sets, the
  // copy streams, a second compute stream and the events that order copies
  // and compute
  static constexpr int kHostSets = 3;
  float *host_ws = nullptr;
  size_t host_ws_bytes = 0;
  cudaStream_t h2d = nullptr, d2h = nullptr, comp2 = nullptr;
  cudaEvent_t ev_start = nullptr, ev_in[kHostSets] = {}, ev_comp[kHostSets] = {},
              ev_out[kHostSets] = {};
  int num_sms = 0;
};
attn_status_t device_state(DeviceState **out);
// Grows the split-key workspace to at least `bytes` (waits for queued work
// before freeing a smaller one).
attn_status_t ensure_split_workspace(DeviceState *ds, size_t bytes);
attn_status_t ensure_bwd_workspace(DeviceState *ds, size_t bytes);
// Dense, non-causal forward: decides whether the last tiles run as key
// halves (when they would fill at most half of the final wave) and, if so,
// sets a.split_rem and the partial buffers.
attn_status_t plan_tail_split(DeviceState *ds, LaunchArgs &a);

// Launches the varlen tile-list builder (one CTA) on `s`.
cudaError_t launch_varlen_schedule(const int *cu_seqlens, int nseq, int total_tokens,
                                   int max_seqlen, int causal, int2 *tiles, int capacity,
                                   int *num_entries, int *status, cudaStream_t s);
attn_status_t ensure_tiles(DeviceState *ds, size_t entries);
long long wait_budget();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace attn
