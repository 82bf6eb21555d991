// Instantiations of the one-tile kernel for attn_fwd on bfloat16 inputs with the
// fp16 copy of V (fp16 P, one P·V product per key block; one key split).
#include "attn_kv_launch.cuh"

namespace ex19 {

cudaError_t launch_kv_pv16(int d, bool out_f32, const KvLaunchArgs& a) {
  if (d == 64)
    return out_f32 ? launch_kv_one<64, true, true, false, true>(a)
                   : launch_kv_one<64, true, false, false, true>(a);
  return out_f32 ? launch_kv_one<128, true, true, false, true>(a)
                 : launch_kv_one<128, true, false, false, true>(a);
}

}  // namespace ex19
