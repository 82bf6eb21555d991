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
  // A programmatic dependent launch (as the decode kernels): the kernel may start its
  // prologue while the previous kernel on the stream finishes, and waits for it
  // (griddepcontrol.wait) before touching global memory or TMEM.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = a.grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, *a.tm_q, *a.tm_k, *a.tm_v, a.p);
}

}  // namespace ex19
