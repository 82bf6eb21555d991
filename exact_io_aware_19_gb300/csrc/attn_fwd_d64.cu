// Instantiations of the attention-forward kernel for head dimension 64.
#include "attn_fwd_launch.cuh"

namespace ex19 {

cudaError_t launch_fwd_d64(bool bf16, bool out_f32, const LaunchArgs& a) {
  if (bf16) return out_f32 ? launch_fwd_one<64, true, true, false>(a) : launch_fwd_one<64, true, false, false>(a);
  return out_f32 ? launch_fwd_one<64, false, true, false>(a) : launch_fwd_one<64, false, false, false>(a);
}

cudaError_t launch_fwd_alt(bool out_f32, const LaunchArgs& a) {
  return out_f32 ? launch_fwd_one<64, false, true, false, true>(a) : launch_fwd_one<64, false, false, false, true>(a);
}

}  // namespace ex19
