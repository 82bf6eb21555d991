// attn_fwd_launch.cuh — launch of one instantiation of the attention-forward kernel
// (included by the translation units that instantiate it).
#pragma once
#include <atomic>

#include "attn_fwd_kernel.cuh"
#include "attn_launch.h"

namespace ex19 {

template <int D, bool BF16, bool OUT_F32, bool PV16, bool ALT = false>
cudaError_t launch_fwd_one(const LaunchArgs& a) {
  auto kern = attn_fwd_sm103_kernel<D, BF16, OUT_F32, PV16, ALT>;
  constexpr int smem = Geometry<D>::kSmemBytes;
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

}  // namespace ex19
