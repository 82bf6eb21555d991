// Instantiations of the backward pass: the D / LSE2 pass, the dQ kernel and the
// dK / dV kernel.
#include <atomic>

#include "attn_bwd_kernel.cuh"
#include "attn_launch.h"

namespace ex19 {
namespace {

template <typename Kern>
cudaError_t set_smem_once(Kern kern, int smem, std::atomic<unsigned long long>& configured) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev < 64) ? (1ull << dev) : 0ull;
  if (bit == 0 || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  return cudaSuccess;
}

template <int D, bool BF16, bool OUT_F32>
cudaError_t launch_bwd_one(const BwdLaunchArgs& a) {
  const bwd::BwdParams& p = a.p;
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.Lpad;
  bwd::attn_bwd_prep<D, BF16><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, a.stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  constexpr int smem = bwd::BwdGeometry<D>::kSmemBytes;
  static std::atomic<unsigned long long> conf_dq{0}, conf_dkdv{0};
  auto kdq = bwd::attn_bwd_dq_kernel<D, BF16, OUT_F32>;
  auto kdkdv = bwd::attn_bwd_dkdv_kernel<D, BF16, OUT_F32>;
  if ((e = set_smem_once(kdq, smem, conf_dq)) != cudaSuccess) return e;
  if ((e = set_smem_once(kdkdv, smem, conf_dkdv)) != cudaSuccess) return e;
  // The dQ and dK / dV kernels are programmatic dependent launches: each may start
  // (barriers, TMEM allocation) as the kernel before it finishes, and waits for it
  // with griddepcontrol.wait before reading global memory.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(bwd::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = a.grid_dq;
  if ((e = cudaLaunchKernelEx(&cfg, kdq, *a.tm_qp, *a.tm_dop, *a.tm_k, *a.tm_v, p)) != cudaSuccess)
    return e;
  cfg.gridDim = a.grid_dkdv;
  return cudaLaunchKernelEx(&cfg, kdkdv, *a.tm_q, *a.tm_do, *a.tm_k, *a.tm_v, *a.tm_lse2, *a.tm_dsum,
                            p);
}

template <int D>
cudaError_t launch_bwd_d(bool bf16, bool out_f32, const BwdLaunchArgs& a) {
  if (bf16) return out_f32 ? launch_bwd_one<D, true, true>(a) : launch_bwd_one<D, true, false>(a);
  return out_f32 ? launch_bwd_one<D, false, true>(a) : launch_bwd_one<D, false, false>(a);
}

}  // namespace

cudaError_t launch_bwd(int d, bool bf16, bool out_f32, const BwdLaunchArgs& a) {
  return (d == 64) ? launch_bwd_d<64>(bf16, out_f32, a) : launch_bwd_d<128>(bf16, out_f32, a);
}

}  // namespace ex19
