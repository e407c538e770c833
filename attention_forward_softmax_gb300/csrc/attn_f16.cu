// attn_f16.cu -- f16 instantiations of the fused attention forward kernel.
#include "attn_launch.cuh"

namespace attn {

attn_status_t launch_attn_f16(const LaunchArgs &a, bool varlen, cudaStream_t s) {
  if (a.d == 128)
    return varlen ? launch_cfg<Cfg<128, Elem::F16, true>>(a, s)
                  : launch_cfg<Cfg<128, Elem::F16, false>>(a, s);
  if (a.d == 64)
    return varlen ? launch_cfg<Cfg<64, Elem::F16, true>>(a, s)
                  : launch_cfg<Cfg<64, Elem::F16, false>>(a, s);
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
