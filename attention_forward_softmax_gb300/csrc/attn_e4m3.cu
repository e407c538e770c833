// attn_e4m3.cu -- e4m3 instantiation of the fused attention forward kernel.
#include "attn_launch.cuh"

namespace attn {

attn_status_t launch_attn_e4m3(const LaunchArgs &a, cudaStream_t s) {
  // d = 64 runs the d = 128 layout: the tensor copies fill the upper 64
  // columns of every Q, K and V row with zeros (outside the tensor), which
  // add nothing to Q K^T and give zero columns of O that are not stored
  if (a.d == 128 || a.d == 64) return launch_cfg<Cfg<128, Elem::E4M3, false>>(a, s);
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
