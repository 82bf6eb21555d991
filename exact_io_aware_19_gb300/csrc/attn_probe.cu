// Launcher of the one-warp bounded-wait probe (tests the timeout path alone).
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"
#include "attn_launch.h"

namespace ex19 {

// One-warp probe of the bounded wait: a barrier nothing completes.
__global__ void wait_probe_kernel(uint32_t* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  WaitCtl wc;
  wc.abort_flag = &abort_flag;
  wc.status = status;
  wc.set_limit(limit_ns);
  wc.unit = 0;
  mbar_wait_warp(smem_u32(&bar), 0, wc, 0x50001);
}


// Element-wise 2^x by the fp32 MUFU instruction and, when y_f16 is given, by the
// packed fp16 one (arguments rounded to fp16 first), for accuracy tests.
__global__ void exp2_probe_kernel(const float* x, float* y_mufu, float* y_f16, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float a = x[i];
  const float b = (i + 1 < n) ? x[i + 1] : 0.f;
  y_mufu[i] = ex2_approx(a);
  if (y_f16 != nullptr) {
    __half2 h = __floats2half2_rn(a, b);
    const uint32_t r = ex2_f16x2(*reinterpret_cast<uint32_t*>(&h));
    y_f16[i] = __half2float(__ushort_as_half(static_cast<unsigned short>(r & 0xFFFFu)));
    if (i + 1 < n) y_f16[i + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(r >> 16)));
  }
  if (i + 1 < n) y_mufu[i + 1] = ex2_approx(b);
}

cudaError_t launch_exp2_probe(const float* x, float* y_mufu, float* y_f16, int n,
                              cudaStream_t stream) {
  const int pairs = (n + 1) / 2;
  exp2_probe_kernel<<<(pairs + 255) / 256, 256, 0, stream>>>(x, y_mufu, y_f16, n);
  return cudaGetLastError();
}

cudaError_t launch_wait_probe(uint32_t* status, unsigned long long limit_ns, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace ex19
