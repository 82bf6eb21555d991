// attn_noalloc.cu — attn_fwd_noalloc: the attention forward for callers that must
// not allocate device memory.
//
// attn_fwd needs a small device workspace (its status word) from the caller. Some
// callers cannot provide one: code that runs where cudaMalloc is forbidden or
// unsafe (inside a custom allocator or memory-pool callback, in a process whose
// device memory is owned by another framework's allocator, or in a tight
// real-time path that must not call into the allocator). This entry point keeps
// that scratch in a fixed, file-scope device array instead, so the call itself
// allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
//
// Costs and limits, stated for the user:
//   * the array is kNoAllocScratchBytes = 256 bytes; every GPU that loads this
//     library holds it until the process exits;
//   * a problem whose workspace need exceeds 256 bytes is rejected with
//     ATTN_ERR_WORKSPACE (no shape needs more today);
//   * all calls on a device share the one array. Each call clears the status word
//     at its start (on the call's stream), so calls that overlap on the GPU — on
//     different streams, or from different threads — race on it; serialise them;
//   * the first call on each device looks up the array's device address with
//     cudaGetSymbolAddress (loading this file's module if needed). Make that first
//     call before any stream capture begins;
//   * a device-side timeout is recorded in this shared status word, which no
//     other entry point reads; callers that need that report should use attn_fwd
//     with their own workspace and attn_fwd_sync_status.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "attn.h"

namespace ex19 {
void set_last_error_detail(const std::string& msg);  // defined in attn_api.cu
}

namespace {

constexpr size_t kNoAllocScratchBytes = 256;
constexpr size_t kStatusWordBytes = 16;

// The scratch of attn_fwd_noalloc (holds the kernel's status word).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on device `dev`, looked up once per device
// with that device current (the caller of attn_fwd_noalloc made it current).
void* scratch_on_device(int dev, cudaError_t* err) {
  static std::mutex mu;
  static void* addr[64] = {};
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      *err = e;
      return nullptr;
    }
    addr[dev] = p;
  }
  *err = cudaSuccess;
  return addr[dev];
}

}  // namespace

extern "C" attn_status_t attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o,
                                          float* lse, int B, int L, int Hq, int Hkv, int d,
                                          int causal, int window_left, float scale,
                                          attn_dtype_t dtype, attn_out_t out_dtype,
                                          void* stream) {
  const size_t need = attn_fwd_workspace_size(B, L, Hq, Hkv, d, causal, window_left);
  if (need == 0) {
    // An invalid shape: attn_fwd reports it (and its detail) before touching memory.
    return attn_fwd(q, k, v, o, lse, B, L, Hq, Hkv, d, causal, window_left, scale, dtype,
                    out_dtype, nullptr, 0, stream);
  }
  if (need > kNoAllocScratchBytes) {
    ex19::set_last_error_detail("this problem needs " + std::to_string(need) +
                                " bytes of scratch; attn_fwd_noalloc holds " +
                                std::to_string(kNoAllocScratchBytes) +
                                " (use attn_fwd with a workspace)");
    return ATTN_ERR_WORKSPACE;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  void* scratch = (e == cudaSuccess) ? scratch_on_device(dev, &e) : nullptr;
  if (scratch == nullptr) {
    ex19::set_last_error_detail(std::string("locating the no-allocation scratch: ") +
                                cudaGetErrorName(e));
    return ATTN_ERR_CUDA;
  }
  // The status word must start at zero (the kernel records only the first error).
  e = cudaMemsetAsync(scratch, 0, kStatusWordBytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    ex19::set_last_error_detail(std::string("clearing the scratch status word: ") +
                                cudaGetErrorName(e));
    return ATTN_ERR_CUDA;
  }
  return attn_fwd(q, k, v, o, lse, B, L, Hq, Hkv, d, causal, window_left, scale, dtype,
                  out_dtype, scratch, kNoAllocScratchBytes, stream);
}
