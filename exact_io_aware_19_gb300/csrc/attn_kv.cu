// Instantiations of the decode-shaped (split-KV) forward and its merge kernel.
#include "attn_kv_launch.cuh"

namespace ex19 {
namespace {

template <int D, bool PAGED>
cudaError_t launch_kv_d(bool bf16, bool out_f32, const KvLaunchArgs& a) {
  if (kv_keys_shape(a.p.q_per_tile, a.p.group)) return launch_kv_keys(D, bf16, PAGED, out_f32, a);
  if (bf16)
    return out_f32 ? launch_kv_one<D, true, true, PAGED>(a) : launch_kv_one<D, true, false, PAGED>(a);
  return out_f32 ? launch_kv_one<D, false, true, PAGED>(a) : launch_kv_one<D, false, false, PAGED>(a);
}

}  // namespace

cudaError_t launch_kv_merge(int d, bool bf16, bool out_f32, const KvLaunchArgs& a) {
  if (d == 64) {
    if (bf16) return out_f32 ? launch_kv_merge_t<64, true, true>(a) : launch_kv_merge_t<64, true, false>(a);
    return out_f32 ? launch_kv_merge_t<64, false, true>(a) : launch_kv_merge_t<64, false, false>(a);
  }
  if (bf16) return out_f32 ? launch_kv_merge_t<128, true, true>(a) : launch_kv_merge_t<128, true, false>(a);
  return out_f32 ? launch_kv_merge_t<128, false, true>(a) : launch_kv_merge_t<128, false, false>(a);
}

cudaError_t launch_kv(int d, bool bf16, bool out_f32, const KvLaunchArgs& a) {
  return (d == 64) ? launch_kv_d<64, false>(bf16, out_f32, a) : launch_kv_d<128, false>(bf16, out_f32, a);
}

cudaError_t launch_kv_paged(int d, bool bf16, bool out_f32, const KvLaunchArgs& a) {
  return (d == 64) ? launch_kv_d<64, true>(bf16, out_f32, a) : launch_kv_d<128, true>(bf16, out_f32, a);
}

}  // namespace ex19
