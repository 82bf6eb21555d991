// Instantiations of the float8 e4m3 forward and of its V transpose.
#include <atomic>

#include "attn_fp8_kernel.cuh"
#include "attn_launch.h"

namespace ex19 {
namespace {

template <bool OUT_F32>
cudaError_t launch_fp8_one(const Fp8LaunchArgs& a) {
  auto kern = fp8::attn_fp8_sm103_kernel<OUT_F32>;
  constexpr int smem = fp8::Fp8Geometry::kSmemBytes;
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
  // Programmatic dependent launch: the prologue (barriers, TMEM allocation) overlaps
  // the end of the V transpose; the kernel waits for it before any global access.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = a.grid;
  cfg.blockDim = dim3(fp8::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, *a.tm_q, *a.tm_k, *a.tm_vt, a.p);
}

}  // namespace

cudaError_t launch_fp8(bool out_f32, const Fp8LaunchArgs& a) {
  const dim3 tgrid((a.Lp + 127) / 128, a.p.Hkv, a.p.B);
  fp8::attn_fp8_transpose_v<<<tgrid, 128, 0, a.stream>>>(a.v, a.vt, a.p.Lk, a.p.Hkv, a.Lp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return out_f32 ? launch_fp8_one<true>(a) : launch_fp8_one<false>(a);
}

}  // namespace ex19
