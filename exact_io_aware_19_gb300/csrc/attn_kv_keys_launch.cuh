// attn_kv_keys_launch.cuh — launch of the keys-on-lanes decode kernel (included by
// the translation units that instantiate it, one per head dimension).
#pragma once
#include <atomic>

#include "attn_kv_keys_kernel.cuh"
#include "attn_launch.h"

namespace ex19 {

template <int D, bool BF16, bool PAGED, int NQ>
cudaError_t launch_keys_one(bool out_f32, const KvLaunchArgs& a) {
  auto kern = kv::attn_kv_keys_kernel<D, BF16, PAGED, NQ>;
  constexpr int smem = kv::KeysGeometry<D>::kSmemBytes;
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
  // A programmatic dependent launch, like the one-tile kernel (see its launch).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = a.grid;
  cfg.blockDim = dim3(kv::kKeysThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // With key splits, items of at most 8 rows merge them in the kernel (the last CTA
  // of each item; the tickets must be in the workspace), so this is the call's only
  // launch; 32-row items are merged by the merge kernel after it.
  if (NQ <= 8 && a.p.splits > 1 && a.p.tickets == nullptr) return cudaErrorInvalidValue;
  e = cudaLaunchKernelEx(&cfg, kern, *a.tm_q, *a.tm_k, *a.tm_v, a.p, out_f32 ? 1 : 0);
  if (e != cudaSuccess || NQ <= 8 || a.p.splits <= 1) return e;
  return launch_kv_merge(D, BF16, out_f32, a);
}

template <int D, bool BF16, bool PAGED>
cudaError_t launch_keys_rows(bool out_f32, const KvLaunchArgs& a) {
  const int rows = a.p.q_per_tile * a.p.group;
  if (rows <= 1) return launch_keys_one<D, BF16, PAGED, 1>(out_f32, a);
  if (rows <= 8) return launch_keys_one<D, BF16, PAGED, 8>(out_f32, a);
  return launch_keys_one<D, BF16, PAGED, 32>(out_f32, a);
}

template <int D>
cudaError_t launch_keys_d(bool bf16, bool paged, bool out_f32, const KvLaunchArgs& a) {
  if (bf16)
    return paged ? launch_keys_rows<D, true, true>(out_f32, a) : launch_keys_rows<D, true, false>(out_f32, a);
  return paged ? launch_keys_rows<D, false, true>(out_f32, a) : launch_keys_rows<D, false, false>(out_f32, a);
}

}  // namespace ex19
