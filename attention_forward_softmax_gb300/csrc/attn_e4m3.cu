// attn_e4m3.cu -- e4m3 instantiation of the fused attention forward kernel.
#include "attn_launch.cuh"

namespace attn {

attn_status_t launch_attn_e4m3(const LaunchArgs &a, cudaStream_t s) {
  if (a.d == 128) return launch_cfg<Cfg<128, Elem::E4M3, false>>(a, s);
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
