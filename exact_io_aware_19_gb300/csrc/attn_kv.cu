// Instantiations of the decode-shaped (split-KV) forward and its merge kernel.
#include "attn_kv_launch.cuh"

namespace ex19 {
namespace {

template <int D, bool PAGED>
cudaError_t launch_kv_d(bool bf16, bool out_f32, const KvLaunchArgs& a) {
  if (bf16)
    return out_f32 ? launch_kv_one<D, true, true, PAGED, false>(a)
                   : launch_kv_one<D, true, false, PAGED, false>(a);
  if constexpr (D == 64) {
    if (kv_decode_mode(D, bf16, a.p.q_per_tile, a.p.group))
      return out_f32 ? launch_kv_one<D, false, true, PAGED, true>(a)
                     : launch_kv_one<D, false, false, PAGED, true>(a);
  }
  return out_f32 ? launch_kv_one<D, false, true, PAGED, false>(a)
                 : launch_kv_one<D, false, false, PAGED, false>(a);
}

}  // namespace

cudaError_t launch_kv(int d, bool bf16, bool out_f32, const KvLaunchArgs& a) {
  return (d == 64) ? launch_kv_d<64, false>(bf16, out_f32, a) : launch_kv_d<128, false>(bf16, out_f32, a);
}

cudaError_t launch_kv_paged(int d, bool bf16, bool out_f32, const KvLaunchArgs& a) {
  return (d == 64) ? launch_kv_d<64, true>(bf16, out_f32, a) : launch_kv_d<128, true>(bf16, out_f32, a);
}

}  // namespace ex19
