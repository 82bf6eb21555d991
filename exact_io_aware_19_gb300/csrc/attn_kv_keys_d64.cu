// Instantiations of the keys-on-lanes decode kernel for head dimension 64, and the
// dispatch over head dimensions.
#include "attn_kv_keys_launch.cuh"

namespace ex19 {

cudaError_t launch_kv_keys_d128(bool bf16, bool paged, bool out_f32, const KvLaunchArgs& a);

cudaError_t launch_kv_keys(int d, bool bf16, bool paged, bool out_f32, const KvLaunchArgs& a) {
  if (a.p.q_per_tile * a.p.group > kv::kKeysRowsMax) return cudaErrorInvalidValue;
  return d == 64 ? launch_keys_d<64>(bf16, paged, out_f32, a) : launch_kv_keys_d128(bf16, paged, out_f32, a);
}

}  // namespace ex19
