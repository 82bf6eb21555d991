// Launcher of the one-warp bounded-wait probe (tests the timeout path alone).
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
  wc.limit_ns = limit_ns;
  wc.unit = 0;
  mbar_wait_warp(smem_u32(&bar), 0, wc, 0x50001);
}


cudaError_t launch_wait_probe(uint32_t* status, unsigned long long limit_ns, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace ex19
