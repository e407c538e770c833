// attn_bf16.cu -- bf16 instantiations of the fused attention forward kernel.
#include "attn_launch.cuh"

namespace attn {

attn_status_t launch_attn_bf16(const LaunchArgs &a, bool varlen, cudaStream_t s) {
  if (a.d == 128)
    return varlen ? launch_cfg<Cfg<128, Elem::BF16, true>>(a, s)
                  : launch_cfg<Cfg<128, Elem::BF16, false>>(a, s);
  if (a.d == 64)
    return varlen ? launch_cfg<Cfg<64, Elem::BF16, true>>(a, s)
                  : launch_cfg<Cfg<64, Elem::BF16, false>>(a, s);
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
