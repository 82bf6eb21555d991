// Instantiations of the keys-on-lanes decode kernel for head dimension 128.
#include "attn_kv_keys_launch.cuh"

namespace ex19 {

cudaError_t launch_kv_keys_d128(bool bf16, bool paged, bool out_f32, const KvLaunchArgs& a) {
  return launch_keys_d<128>(bf16, paged, out_f32, a);
}

}  // namespace ex19
