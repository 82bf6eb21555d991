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
//     ATTN_ERR_WORKSPACE (no shape needs more: bfloat16 inputs run attn_fwd's
//     split-weight path, which makes no copy of V);
//   * all calls on a device share the one array. Each call clears the status word
//     (on the call's stream, after its arguments are validated), so calls that
//     overlap on the GPU — on different streams, or from different threads — race
//     on it; serialise them;
//   * the first call on each device, and the first after that device's context was
//     destroyed and created again (cudaDeviceReset), looks up the array's device
//     address with cudaGetSymbolAddress (loading this file's module if needed).
//     Make that first call before any stream capture begins;
//   * a device-side timeout is recorded in this shared status word, which no
//     other entry point reads; callers that need that report should use attn_fwd
//     with their own workspace and attn_fwd_sync_status.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <string>

#include "attn.h"

namespace ex19 {
void set_last_error_detail(const std::string& msg);  // defined in attn_api.cu
attn_status_t current_sm103_device(int* dev);        // defined in attn_api.cu
attn_status_t fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int L, int Hq, int Hkv, int d, int causal, int window_left, float scale,
                       attn_dtype_t dtype, attn_out_t out_dtype, void* workspace,
                       size_t workspace_bytes, void* stream, size_t clear_status_bytes);
}

namespace {

constexpr size_t kNoAllocScratchBytes = 256;
constexpr size_t kStatusWordBytes = 16;

// The scratch of attn_fwd_noalloc (holds the kernel's status word).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Driver calls that identify the current context (cuCtxGetId gives an id that is
// never reused within the process, so a context created again after a reset gets
// a new one).
struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxFns& ctx_fns() {
  static std::once_flag once;
  static CtxFns fns;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return fns;
}

// Id of the calling thread's current context, or 0 when there is none (or the
// driver cannot say).
unsigned long long current_ctx_id() {
  const CtxFns& f = ctx_fns();
  if (f.get_current == nullptr || f.get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  return f.get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of g_noalloc_scratch on device `dev` (current), cached per device
// and context: a context destroyed and created again (cudaDeviceReset) may load
// the module at another address, so a new context id triggers a new lookup.
void* scratch_on_device(int dev, cudaError_t* err) {
  static std::mutex mu;
  static void* addr[64] = {};
  static unsigned long long ctx_of[64] = {};
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long id = current_ctx_id();
  if (addr[dev] == nullptr || id == 0 || id != ctx_of[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      cudaGetLastError();  // leave no sticky error behind for unrelated calls
      addr[dev] = nullptr;
      *err = e;
      return nullptr;
    }
    addr[dev] = p;
    // the lookup made the primary context current if none was
    ctx_of[dev] = (id != 0) ? id : current_ctx_id();
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
  // The least workspace attn_fwd accepts (the status word; fp16's full size). With
  // bfloat16 inputs so small a workspace runs the split-weight path, which needs no
  // copy of V.
  const size_t need = attn_fwd_workspace_size(B, L, Hq, Hkv, d, causal, window_left, ATTN_FP16);
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
  const attn_status_t st = ex19::current_sm103_device(&dev);  // no image for other devices
  if (st != ATTN_OK) return st;
  cudaError_t e = cudaSuccess;
  void* scratch = scratch_on_device(dev, &e);
  if (scratch == nullptr) {
    ex19::set_last_error_detail(std::string("locating the no-allocation scratch: ") +
                                cudaGetErrorName(e));
    return ATTN_ERR_CUDA;
  }
  // The status word must start at zero (the kernel records only the first error);
  // attn_fwd's checks run first, so a rejected call enqueues nothing.
  return ex19::fwd_impl(q, k, v, o, lse, B, L, Hq, Hkv, d, causal, window_left, scale, dtype,
                        out_dtype, scratch, kNoAllocScratchBytes, stream, kStatusWordBytes);
}
