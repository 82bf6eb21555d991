// Instantiations of the attention-forward kernel for head dimension 128.
#include "attn_fwd_launch.cuh"

namespace ex19 {

cudaError_t launch_fwd_d128(bool bf16, bool out_f32, const LaunchArgs& a) {
  if (bf16) return out_f32 ? launch_fwd_one<128, true, true, false>(a) : launch_fwd_one<128, true, false, false>(a);
  return out_f32 ? launch_fwd_one<128, false, true, false>(a) : launch_fwd_one<128, false, false, false>(a);
}

}  // namespace ex19
