// attn_bias.cu -- 16-bit instantiations of the fused attention forward kernel
// with an additive fp32 score bias (dense layout).
#include "attn_launch.cuh"

namespace attn {

attn_status_t launch_attn_bias(const LaunchArgs &a, bool bf16, cudaStream_t s) {
  if (a.d == 128)
    return bf16 ? launch_cfg<Cfg<128, Elem::BF16, false, true>>(a, s)
                : launch_cfg<Cfg<128, Elem::F16, false, true>>(a, s);
  if (a.d == 64)
    return bf16 ? launch_cfg<Cfg<64, Elem::BF16, false, true>>(a, s)
                : launch_cfg<Cfg<64, Elem::F16, false, true>>(a, s);
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
