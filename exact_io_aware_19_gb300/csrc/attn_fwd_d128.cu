// Instantiations of the attention-forward kernel for head dimension 128.
#include <atomic>

#include "attn_fwd_kernel.cuh"
#include "attn_launch.h"

namespace ex19 {
namespace {

template <bool BF16, bool OUT_F32>
cudaError_t launch_one(const LaunchArgs& a) {
  auto kern = attn_fwd_sm103_kernel<128, BF16, OUT_F32>;
  constexpr int smem = Geometry<128>::kSmemBytes;
  static std::atomic<unsigned long long> configured{0};  // one bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev < 64) ? (1ull << dev) : 0ull;
  if (bit == 0 || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  kern<<<a.grid, kThreads, smem, a.stream>>>(*a.tm_q, *a.tm_k, *a.tm_v, a.p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_d128(bool bf16, bool out_f32, const LaunchArgs& a) {
  if (bf16) return out_f32 ? launch_one<true, true>(a) : launch_one<true, false>(a);
  return out_f32 ? launch_one<false, true>(a) : launch_one<false, false>(a);
}

}  // namespace ex19
