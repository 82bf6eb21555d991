// attn_kv_launch.cuh — launch of one instantiation of the one-tile (split-KV)
// kernel and, when the call has several key splits, its merge kernel (included by the
// translation units that instantiate them).
#pragma once
#include <atomic>

#include "attn_kv_kernel.cuh"
#include "attn_launch.h"

namespace ex19 {

// The merge of a call's key splits (a programmatic dependent launch after the split
// kernel): one CTA per row when the call has at most one row per SM (decode: many
// splits per row), one warp per row otherwise.
template <int D, bool BF16, bool OUT_F32>
cudaError_t launch_kv_merge_t(const KvLaunchArgs& a) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int sms = 148;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = a.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const long long rows = static_cast<long long>(a.p.B) * a.p.Hq * a.p.Lq;
  if (rows <= sms) {  // few rows (decode): one CTA per row
    cfg.gridDim = dim3(static_cast<unsigned>(rows));
    return cudaLaunchKernelEx(&cfg, kv::attn_kv_merge_kernel<D, BF16, OUT_F32, 8>, a.p);
  }
  cfg.gridDim = dim3(static_cast<unsigned>((rows + 7) / 8));  // many rows: one warp per row
  return cudaLaunchKernelEx(&cfg, kv::attn_kv_merge_kernel<D, BF16, OUT_F32, 1>, a.p);
}

template <int D, bool BF16, bool OUT_F32, bool PAGED, bool PV16 = false>
cudaError_t launch_kv_one(const KvLaunchArgs& a) {
  auto kern = kv::attn_kv_sm103_kernel<D, BF16, OUT_F32, PAGED, PV16>;
  if (PV16 && a.p.splits != 1) return cudaErrorInvalidValue;  // attn_fwd's path: one key split
  constexpr int smem = kv::KvGeometry<D>::kSmemBytes;
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
  // Both kernels are programmatic dependent launches: each may start while the
  // previous kernel on the stream finishes, and waits for it (griddepcontrol.wait)
  // before touching global memory. The split kernel's prologue (barriers, TMEM
  // allocation, tensor-map prefetch) and the merge's launch overlap the kernel
  // before them.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = a.grid;
  cfg.blockDim = dim3(kv::KvRoles::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, *a.tm_q, *a.tm_k, *a.tm_v, a.p);
  if constexpr (PV16) {
    return e;  // one key split (checked above): no merge
  } else {
    if (e != cudaSuccess || a.p.splits <= 1) return e;
    return launch_kv_merge(D, BF16, OUT_F32, a);
  }
}

}  // namespace ex19
