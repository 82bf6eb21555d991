// Instantiations of the attention-forward kernel for bfloat16 inputs with the fp16
// copy of V (fp16 P, one P·V product per key block).
#include "attn_fwd_launch.cuh"

namespace ex19 {

cudaError_t launch_fwd_pv16(int d, bool out_f32, const LaunchArgs& a) {
  if (d == 64) return out_f32 ? launch_fwd_one<64, true, true, true>(a) : launch_fwd_one<64, true, false, true>(a);
  return out_f32 ? launch_fwd_one<128, true, true, true>(a) : launch_fwd_one<128, true, false, true>(a);
}

}  // namespace ex19
