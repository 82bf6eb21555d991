// attn_api.cu — the C ABI declared in include/attn.h: argument validation, TMA
// tensor maps, grid sizing and launch. Host code only; no device allocation.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "attn.h"
#include "attn_launch.h"
#include "vscale.cuh"

namespace {

// status word (16 B) and the persistent kernel's unit counter (at byte 64), padded to
// 256 bytes
constexpr size_t kWorkspaceBytes = 256;
constexpr size_t kSchedOffset = 64;
constexpr unsigned long long kDefaultWaitLimitNs = 4000000000ull;
constexpr int kUnitRows = 256;           // query rows per kernel work unit

thread_local std::string g_detail;
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<int> g_path_policy{ATTN_PATH_AUTO};

attn_status_t fail(attn_status_t s, const std::string& msg) {
  g_detail = msg;
  return s;
}

attn_status_t cuda_fail(const char* what, cudaError_t e) {
  return fail(ATTN_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" +
                                 cudaGetErrorString(e) + ")");
}

struct DeviceInfo {
  int sms = 0, major = 0, minor = 0;
};

bool device_info(int dev, DeviceInfo* out, cudaError_t* err) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return false;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev]) {
    DeviceInfo d;
    cudaError_t e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) {
      *err = e;
      return false;
    }
    cache[dev] = d;
    have[dev] = true;
  }
  *out = cache[dev];
  return true;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn(cudaError_t* err) {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static cudaError_t status = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                              cudaEnableDefault, &q);
    if (status == cudaSuccess && q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    } else if (status == cudaSuccess) {
      status = cudaErrorSymbolNotFound;
    }
  });
  *err = status;
  return fn;
}

// Tensor map over a [B, L, H, d] 16-bit tensor. Dimensions are listed innermost
// first with increasing strides (d, H, L, B); the box is 64 elements (128 bytes,
// one swizzle span) of d, box_h heads, box_l rows, 1 batch.
bool make_tensor_map(CUtensorMap* map, const void* ptr, bool bf16, int B, int L, int H, int d,
                     std::string* why, int box_h = 1, int box_l = 128) {
  cudaError_t err;
  auto encode = encode_fn(&err);
  if (encode == nullptr) {
    *why = std::string("cuTensorMapEncodeTiled unavailable: ") + cudaGetErrorName(err);
    return false;
  }
  const cuuint64_t e = 2;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)d * e, (cuuint64_t)H * d * e, (cuuint64_t)L * H * d * e};
  cuuint32_t box[4] = {64, (cuuint32_t)box_h, (cuuint32_t)box_l, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                      4, const_cast<void*>(ptr), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
    return false;
  }
  return true;
}

// Tensor map over a 4-D tensor of bytes (float8 data): dims innermost first, with
// the byte strides of dims 1-3, the box and the swizzle mode.
bool make_tensor_map_u8(CUtensorMap* map, const void* ptr, const cuuint64_t (&dims)[4],
                        const cuuint64_t (&strides)[3], const cuuint32_t (&box)[4],
                        CUtensorMapSwizzle swizzle, std::string* why) {
  cudaError_t err;
  auto encode = encode_fn(&err);
  if (encode == nullptr) {
    *why = std::string("cuTensorMapEncodeTiled unavailable: ") + cudaGetErrorName(err);
    return false;
  }
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled (float8) failed with CUresult " + std::to_string((int)r);
    return false;
  }
  return true;
}

// 2-D tensor map over float32 rows [rows, cols] (cols contiguous), boxes of
// box_cols x 1, no swizzle.
bool make_tensor_map_f32_rows(CUtensorMap* map, const void* ptr, int rows, int cols, int box_cols,
                              std::string* why) {
  cudaError_t err;
  auto encode = encode_fn(&err);
  if (encode == nullptr) {
    *why = std::string("cuTensorMapEncodeTiled unavailable: ") + cudaGetErrorName(err);
    return false;
  }
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, 1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled (float32 rows) failed with CUresult " + std::to_string((int)r);
    return false;
  }
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The pointer must be device (or managed) memory of device `dev`.
bool is_device_ptr(const void* p, int dev, std::string* why, const char* name) {
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *why = std::string(name) + ": cudaPointerGetAttributes failed";
    return false;
  }
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) {
    *why = std::string(name) + " is not device memory";
    return false;
  }
  if (at.type == cudaMemoryTypeDevice && at.device != dev) {
    *why = std::string(name) + " lives on device " + std::to_string(at.device) +
           ", current device is " + std::to_string(dev);
    return false;
  }
  return true;
}

// Shape checks shared by attn_fwd and attn_fwd_workspace_size.
attn_status_t check_shape(int B, int L, int Hq, int Hkv, int d, int causal, int window_left) {
  if (B < 1 || L < 1 || Hq < 1 || Hkv < 1)
    return fail(ATTN_ERR_INVALID_ARG, "B, L, Hq and Hkv must all be >= 1");
  if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "Hq must be a multiple of Hkv");
  if (d < 1) return fail(ATTN_ERR_INVALID_ARG, "d must be >= 1");
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "d must be 64 or 128");
  if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (window_left < -1) return fail(ATTN_ERR_INVALID_ARG, "window_left must be >= -1");
  if (window_left >= 0 && !causal)
    return fail(ATTN_ERR_UNSUPPORTED, "a left window is only supported with causal = 1");
  const long long rows = (long long)B * Hq * L;
  if (rows >= (1LL << 31)) return fail(ATTN_ERR_INVALID_ARG, "B * Hq * L must be < 2^31");
  return ATTN_OK;
}

// attn_fwd's workspace: the status word; with bfloat16 inputs also the heads' largest
// |v| ([B, Hkv] u32, padded to 256 bytes) and the fp16 copy of V ([B, L, Hkv, d]).
size_t fwd_vmax_bytes(int B, int Hkv) { return ((size_t)B * Hkv * 4 + 255) / 256 * 256; }
size_t fwd_workspace_bytes(int B, int L, int Hkv, int d, attn_dtype_t dtype) {
  if (dtype != ATTN_BF16) return kWorkspaceBytes;
  return kWorkspaceBytes + fwd_vmax_bytes(B, Hkv) + (size_t)2 * B * L * Hkv * d;
}

// ---------------------------------------------------------------- decode shapes
constexpr int kKvMaxSplits = 256;

attn_status_t check_kv_shape(int B, int Lq, int Lk, int Hq, int Hkv, int d, int causal,
                             int window_left) {
  if (B < 1 || Lq < 1 || Lk < 1 || Hq < 1 || Hkv < 1)
    return fail(ATTN_ERR_INVALID_ARG, "B, Lq, Lk, Hq and Hkv must all be >= 1");
  if (Lq > Lk) return fail(ATTN_ERR_INVALID_ARG, "Lq must be <= Lk (queries are the last Lq positions)");
  if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "Hq must be a multiple of Hkv");
  if (Hq / Hkv > 128)
    return fail(ATTN_ERR_UNSUPPORTED, "at most 128 query heads may share one K/V head");
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "d must be 64 or 128");
  if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (window_left < -1) return fail(ATTN_ERR_INVALID_ARG, "window_left must be >= -1");
  if (window_left >= 0 && !causal)
    return fail(ATTN_ERR_UNSUPPORTED, "a left window is only supported with causal = 1");
  if ((long long)B * Hq * Lq >= (1LL << 31) || (long long)B * Hkv * Lk >= (1LL << 31))
    return fail(ATTN_ERR_INVALID_ARG, "B * Hq * Lq and B * Hkv * Lk must be < 2^31");
  return ATTN_OK;
}

struct KvPlan {
  int group, q_per_tile, row_tiles, items;  // items = B * Hkv * row_tiles
  int max_blocks;                           // key blocks of the largest row tile
};

KvPlan kv_plan(int B, int Lq, int Lk, int Hq, int Hkv, int causal, int window_left) {
  KvPlan k;
  k.group = Hq / Hkv;
  k.q_per_tile = std::min(Lq, 128 / k.group);
  k.row_tiles = (Lq + k.q_per_tile - 1) / k.q_per_tile;
  k.items = B * Hkv * k.row_tiles;
  const int nblk = (Lk + 127) / 128;
  k.max_blocks = 0;
  for (int rt = 0; rt < k.row_tiles; ++rt) {
    const int i0 = rt * k.q_per_tile, i1 = std::min(Lq, i0 + k.q_per_tile);
    const int off = Lk - Lq;
    const int hi = causal ? (off + i1 - 1) / 128 + 1 : nblk;
    const int lo = window_left >= 0 ? std::max(0, off + i0 - window_left) / 128 : 0;
    k.max_blocks = std::max(k.max_blocks, hi - lo);
  }
  return k;
}

// Splits that fill the SMs with one wave of CTAs (one per SM), keeping at least 2 key
// blocks per split and at most kKvMaxSplits.
int kv_auto_splits(const KvPlan& k, int sms) {
  int s = std::max(1, sms / std::max(1, k.items));
  s = std::min(s, std::max(1, k.max_blocks / 2));
  return std::min(s, kKvMaxSplits);
}

// The decode workspace: the status word, then (splits > 1) the partial LSEs, the
// partial outputs and one merge ticket (8 bytes) per work item.
size_t kv_lse_part_bytes(size_t rows, int splits) { return ((size_t)splits * rows * 4 + 255) / 256 * 256; }

size_t kv_workspace_bytes(int B, int Lq, int Hq, int d, int splits, int items) {
  if (splits <= 1) return kWorkspaceBytes;
  const size_t rows = (size_t)B * Hq * Lq;
  const size_t ticket_bytes = ((size_t)items * 8 + 255) / 256 * 256;
  return kWorkspaceBytes + kv_lse_part_bytes(rows, splits) + (size_t)splits * rows * d * 4 + ticket_bytes;
}

// The tag of a call's merge tickets (kept in bits 9 and up of a ticket word). Each call
// takes the next value of a process-wide counter that starts from the wall clock in
// microseconds, so a tag differs from those of earlier calls and, with all but
// negligible probability, from whatever a fresh workspace holds.
unsigned long long next_ticket_base() {
  static std::atomic<unsigned long long> next{static_cast<unsigned long long>(
      std::chrono::duration_cast<std::chrono::microseconds>(
          std::chrono::system_clock::now().time_since_epoch()).count())};
  const unsigned long long tag = next.fetch_add(1) & ((1ull << 55) - 1);
  return tag << 9;
}

int current_sms(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  DeviceInfo info;
  if (e != cudaSuccess || !device_info(dev, &info, &e)) {
    cudaGetLastError();
    return -1;
  }
  *sms = info.sms;
  return 0;
}

// Paged K/V cache description (attn_fwd_kv_paged); null for the dense entry point.
struct PagedArgs {
  const int32_t* block_table;
  const int32_t* seq_lens;
  int page_size, num_pages, max_pages;
};

// attn_fwd_kv and attn_fwd_kv_paged: validation, plan, tensor maps and launch. For
// the paged call k and v are the caches and Lk is the maximum sequence length.
attn_status_t kv_run(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Lq, int Lk, int Hq, int Hkv, int d, int causal, int window_left,
                     float scale, attn_dtype_t dtype, attn_out_t out_dtype, int num_splits,
                     void* workspace, size_t workspace_bytes, void* stream,
                     const PagedArgs* paged) {
  g_detail.clear();
  attn_status_t st = check_kv_shape(B, Lq, Lk, Hq, Hkv, d, causal, window_left);
  if (st != ATTN_OK) return st;
  if (num_splits < 0 || num_splits > kKvMaxSplits)
    return fail(ATTN_ERR_INVALID_ARG, "num_splits must be in [0, 256]");
  if (!std::isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale must be finite");
  if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return fail(ATTN_ERR_INVALID_ARG, "bad dtype");
  if (out_dtype != ATTN_OUT_SAME && out_dtype != ATTN_OUT_FP32)
    return fail(ATTN_ERR_INVALID_ARG, "bad out_dtype");
  if (!q || !k || !v || !o) return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be non-null");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  if (paged) {
    const int ps = paged->page_size;
    if (ps != 8 && ps != 16 && ps != 32 && ps != 64 && ps != 128)
      return fail(ATTN_ERR_UNSUPPORTED, "page_size must be 8, 16, 32, 64 or 128");
    if (paged->num_pages < 1 || (long long)paged->num_pages * ps >= (1LL << 31))
      return fail(ATTN_ERR_INVALID_ARG, "num_pages must be >= 1 and num_pages * page_size < 2^31");
    if (paged->max_pages < (Lk + ps - 1) / ps)
      return fail(ATTN_ERR_INVALID_ARG, "max_pages_per_seq must cover max_seq_len");
    if (!paged->block_table || !paged->seq_lens)
      return fail(ATTN_ERR_INVALID_ARG, "block_table and seq_lens must be non-null");
    if (!aligned(paged->block_table, 4) || !aligned(paged->seq_lens, 4))
      return fail(ATTN_ERR_INVALID_ARG, "block_table and seq_lens must be 4-byte aligned");
  }
  if (!workspace) return fail(ATTN_ERR_WORKSPACE, "workspace must be non-null");
  if (!aligned(workspace, 16)) return fail(ATTN_ERR_WORKSPACE, "workspace must be 16-byte aligned");
  const KvPlan plan = kv_plan(B, Lq, Lk, Hq, Hkv, causal, window_left);
  if (num_splits > 0 && workspace_bytes < kv_workspace_bytes(B, Lq, Hq, d, num_splits, plan.items))
    return fail(ATTN_ERR_WORKSPACE, "workspace smaller than attn_fwd_kv_workspace_size()");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  DeviceInfo info;
  if (!device_info(dev, &info, &e)) return cuda_fail("cudaDeviceGetAttribute", e);
  if (info.major != 10 || info.minor != 3)
    return fail(ATTN_ERR_UNSUPPORTED, "needs a compute capability 10.3 device (GB300), found " +
                                          std::to_string(info.major) + "." +
                                          std::to_string(info.minor));
  const int splits = num_splits ? num_splits : kv_auto_splits(plan, info.sms);
  if (workspace_bytes < kv_workspace_bytes(B, Lq, Hq, d, splits, plan.items))
    return fail(ATTN_ERR_WORKSPACE, "workspace smaller than attn_fwd_kv_workspace_size()");
  if ((long long)plan.items * splits >= (1LL << 31))
    return fail(ATTN_ERR_INVALID_ARG, "too many work items");
  std::string why;
  const void* ptrs[8] = {q, k, v, o, workspace, lse, paged ? paged->block_table : nullptr,
                         paged ? paged->seq_lens : nullptr};
  const char* names[8] = {"q", "k", "v", "o", "workspace", "lse", "block_table", "seq_lens"};
  for (int i = 0; i < 8; ++i)
    if (ptrs[i] && !is_device_ptr(ptrs[i], dev, &why, names[i]))
      return fail(ATTN_ERR_INVALID_ARG, why);

  const bool bf16 = dtype == ATTN_BF16;
  CUtensorMap tm_q, tm_k, tm_v;
  bool maps_ok = make_tensor_map(&tm_q, q, bf16, B, Lq, Hq, d, &why, plan.group, plan.q_per_tile);
  if (maps_ok && paged) {
    // the caches as one sequence of num_pages * page_size rows; one box = one page
    const int rows = paged->num_pages * paged->page_size;
    maps_ok = make_tensor_map(&tm_k, k, bf16, 1, rows, Hkv, d, &why, 1, paged->page_size) &&
              make_tensor_map(&tm_v, v, bf16, 1, rows, Hkv, d, &why, 1, paged->page_size);
  } else if (maps_ok) {
    maps_ok = make_tensor_map(&tm_k, k, bf16, B, Lk, Hkv, d, &why) &&
              make_tensor_map(&tm_v, v, bf16, B, Lk, Hkv, d, &why);
  }
  if (!maps_ok) return fail(ATTN_ERR_CUDA, why);

  ex19::KvLaunchArgs a = {};
  a.tm_q = &tm_q;
  a.tm_k = &tm_k;
  a.tm_v = &tm_v;
  ex19::KvParams& p = a.p;
  p.o = o;
  p.lse = lse;
  p.status = static_cast<uint32_t*>(workspace);
  const size_t rows = (size_t)B * Hq * Lq;
  if (splits > 1) {
    char* base = static_cast<char*>(workspace) + kWorkspaceBytes;
    const size_t lse_bytes = kv_lse_part_bytes(rows, splits);
    p.lse_part = reinterpret_cast<float*>(base);
    p.o_part = reinterpret_cast<float*>(base + lse_bytes);
    p.tickets = reinterpret_cast<unsigned long long*>(base + lse_bytes + (size_t)splits * rows * d * 4);
    p.ticket_base = next_ticket_base();
  }
  p.B = B;
  p.Lq = Lq;
  p.Lk = Lk;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = plan.group;
  p.causal = causal;
  p.window_left = window_left;
  p.window_right = -1;
  p.score_log2 = std::fabs(scale) * 1.4426950408889634f;
  p.negate_scores = scale < 0.f ? 1 : 0;
  p.q_per_tile = plan.q_per_tile;
  p.row_tiles = plan.row_tiles;
  p.splits = splits;
  p.wait_limit_ns = g_wait_limit_ns.load();
  if (paged) {
    p.block_table = paged->block_table;
    p.seq_lens = paged->seq_lens;
    p.page_size = paged->page_size;
    p.max_pages = paged->max_pages;
    p.num_pages = paged->num_pages;
  }
  a.grid = plan.items * splits;
  a.stream = static_cast<cudaStream_t>(stream);
  const bool out_f32 = out_dtype == ATTN_OUT_FP32;
  e = paged ? ex19::launch_kv_paged(d, bf16, out_f32, a) : ex19::launch_kv(d, bf16, out_f32, a);
  if (e != cudaSuccess) return cuda_fail("kernel launch", e);
  return ATTN_OK;
}

// The square problem (validated by the caller) on the one-tile kernel: Lq = Lk = L,
// one key split, so no partial results and no merge.
attn_status_t launch_square_as_kv(const void* q, const void* k, const void* v, void* o,
                                  float* lse, int B, int L, int Hq, int Hkv, int d, int causal,
                                  int window_left, int window_right, float scale, bool bf16,
                                  bool out_f32, void* workspace, void* stream,
                                  const void* v16 = nullptr, const uint32_t* vmax = nullptr) {
  const KvPlan plan = kv_plan(B, L, L, Hq, Hkv, causal, window_left);
  if (plan.group > 128)
    return fail(ATTN_ERR_UNSUPPORTED, "at most 128 query heads may share one K/V head");
  std::string why;
  CUtensorMap tm_q, tm_k, tm_v;
  if (!make_tensor_map(&tm_q, q, bf16, B, L, Hq, d, &why, plan.group, plan.q_per_tile) ||
      !make_tensor_map(&tm_k, k, bf16, B, L, Hkv, d, &why) ||
      !(v16 ? make_tensor_map(&tm_v, v16, false, B, L, Hkv, d, &why)
            : make_tensor_map(&tm_v, v, bf16, B, L, Hkv, d, &why)))
    return fail(ATTN_ERR_CUDA, why);
  ex19::KvLaunchArgs a = {};
  a.tm_q = &tm_q;
  a.tm_k = &tm_k;
  a.tm_v = &tm_v;
  ex19::KvParams& p = a.p;
  p.o = o;
  p.lse = lse;
  p.status = static_cast<uint32_t*>(workspace);
  p.o_part = nullptr;
  p.lse_part = nullptr;
  p.vmax = vmax;
  p.B = B;
  p.Lq = L;
  p.Lk = L;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = plan.group;
  p.causal = causal;
  p.window_left = window_left;
  p.window_right = window_right;
  p.score_log2 = std::fabs(scale) * 1.4426950408889634f;
  p.negate_scores = scale < 0.f ? 1 : 0;
  p.q_per_tile = plan.q_per_tile;
  p.row_tiles = plan.row_tiles;
  p.splits = 1;
  p.wait_limit_ns = g_wait_limit_ns.load();
  a.grid = plan.items;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (v16) {
    e = ex19::launch_v_to_f16(v, const_cast<void*>(v16), const_cast<uint32_t*>(vmax), B, L, Hkv, d,
                              a.stream);
    if (e != cudaSuccess) return cuda_fail("the fp16 copy of V", e);
    e = ex19::launch_kv_pv16(d, out_f32, a);
  } else {
    e = ex19::launch_kv(d, bf16, out_f32, a);
  }
  if (e != cudaSuccess) return cuda_fail("kernel launch", e);
  return ATTN_OK;
}

}  // namespace

namespace ex19 {
// Lets other translation units of the library set the detail string that
// attn_last_error_detail() returns to the calling thread.
void set_last_error_detail(const std::string& msg) { g_detail = msg; }

// The current device, if it is a compute capability 10.3 device; otherwise the
// status attn_fwd returns for it (with its detail).
attn_status_t current_sm103_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  DeviceInfo info;
  if (!device_info(*dev, &info, &e)) return cuda_fail("cudaDeviceGetAttribute", e);
  if (info.major != 10 || info.minor != 3)
    return fail(ATTN_ERR_UNSUPPORTED, "needs a compute capability 10.3 device (GB300), found " +
                                          std::to_string(info.major) + "." +
                                          std::to_string(info.minor));
  return ATTN_OK;
}

// attn_fwd, optionally clearing the first `clear_status_bytes` of the workspace on
// the call's stream once every argument has been validated (attn_fwd passes 0).
attn_status_t fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int L, int Hq, int Hkv, int d, int causal, int window_left, float scale,
                       attn_dtype_t dtype, attn_out_t out_dtype, void* workspace,
                       size_t workspace_bytes, void* stream, size_t clear_status_bytes) {
  g_detail.clear();
  attn_status_t st = check_shape(B, L, Hq, Hkv, d, causal, window_left);
  if (st != ATTN_OK) return st;
  if (!std::isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale must be finite");
  if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return fail(ATTN_ERR_INVALID_ARG, "bad dtype");
  if (out_dtype != ATTN_OUT_SAME && out_dtype != ATTN_OUT_FP32)
    return fail(ATTN_ERR_INVALID_ARG, "bad out_dtype");
  if (!q || !k || !v || !o) return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be non-null");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  if (!workspace) return fail(ATTN_ERR_WORKSPACE, "workspace must be non-null");
  if (!aligned(workspace, 16)) return fail(ATTN_ERR_WORKSPACE, "workspace must be 16-byte aligned");
  if (workspace_bytes < kWorkspaceBytes)
    return fail(ATTN_ERR_WORKSPACE, "workspace smaller than attn_fwd_workspace_size()");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  DeviceInfo info;
  if (!device_info(dev, &info, &e)) return cuda_fail("cudaDeviceGetAttribute", e);
  if (info.major != 10 || info.minor != 3)
    return fail(ATTN_ERR_UNSUPPORTED, "needs a compute capability 10.3 device (GB300), found " +
                                          std::to_string(info.major) + "." +
                                          std::to_string(info.minor));
  std::string why;
  const void* ptrs[6] = {q, k, v, o, workspace, lse};
  const char* names[6] = {"q", "k", "v", "o", "workspace", "lse"};
  for (int i = 0; i < 6; ++i)
    if (ptrs[i] && !is_device_ptr(ptrs[i], dev, &why, names[i]))
      return fail(ATTN_ERR_INVALID_ARG, why);
  if (clear_status_bytes > 0) {  // the caller's status word starts at zero (after validation)
    e = cudaMemsetAsync(workspace, 0, clear_status_bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("clearing the status word", e);
  }

  const bool bf16 = dtype == ATTN_BF16;
  const bool out_f32 = out_dtype == ATTN_OUT_FP32;
  // bfloat16 inputs with the full workspace: P·V in fp16 against a per-head scaled
  // fp16 copy of V (one product per key block instead of the split P's two). A
  // workspace of only the status word (attn_fwd_noalloc's) keeps the split P.
  const bool pv16 = bf16 && workspace_bytes >= fwd_workspace_bytes(B, L, Hkv, d, dtype);
  uint32_t* vmax = nullptr;
  void* v16 = nullptr;
  if (pv16) {  // written by launch_v_to_f16 right before the attention kernel
    vmax = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + kWorkspaceBytes);
    v16 = static_cast<char*>(workspace) + kWorkspaceBytes + fwd_vmax_bytes(B, Hkv);
  }
  const int num_units = B * Hq * ((L + kUnitRows - 1) / kUnitRows);
  // Problems with at most half as many 256-row units as SMs leave most SMs idle in
  // the persistent two-tile kernel; the one-tile kernel (the decode-shaped path with
  // Lq = Lk and one key split) runs 128-row tiles, twice as many CTAs. Under a causal
  // mask the work per tile grows with its position, and the persistent kernel's time
  // is then set by its longest unit (the last two tiles, all key blocks, one after
  // another); the one-tile kernel starts the longest tiles first and spreads the
  // rest, which wins up to one unit per SM (measured at L = 8192, 4 heads: 72 against
  // 97 µs; at twice that the persistent kernel's throughput wins).
  // With the split bf16 P (two P·V products per block) the persistent kernel keeps P
  // over S, so a tile's next S product waits for both; the one-tile kernel
  // double-buffers S and runs two softmax threads per row. Under a left window (a few
  // dozen key blocks per tile, two of them masked) it wins while the K/V its keys
  // span stays near L2 (it reads each K/V block for 128 rows, not 256): measured on
  // one GB300, window 4096 4x16x32768 d = 128 bf16 4.83 against 4.99 ms; causal
  // without a window the persistent kernel wins (GQA 32/8 d = 128 L = 16384 2.03
  // against 2.16 ms). With fp16 P (one P·V product) the persistent kernel wins both
  // (3.60 against 4.14 ms, 1.55 against 1.69 ms).
  const int policy = g_path_policy.load();
  const bool few_units = causal ? num_units <= info.sms : 2 * num_units <= info.sms;
  const bool split_p = bf16 && !pv16;
  const int kv_span = (window_left >= 0) ? std::min(L, window_left + 128) : L;
  const double kv_bytes = 4.0 * B * Hkv * static_cast<double>(kv_span) * d;  // K and V, 2 B each
  const bool tiles_win = split_p && window_left >= 0 && kv_bytes <= 192.0 * 1024 * 1024;
  // The alternating mode (one 128-row tile per unit, the two pipelines on alternate
  // key blocks) halves the longest tile's chain; its smaller units also balance the
  // causal triangle better. Measured on one GB300 (causal 4 heads, fp16, d = 64, CUDA
  // events, L2 flushed), against the one-tile kernel below one unit per SM and the
  // two-tile kernel with dynamic scheduling above: L = 2048 27.7 -> 22.1 us, 4096 35.5
  // -> 31.4 us, 8192 90 (61 on the one-tile kernel) -> 52 us, 16384 171 -> 164 us,
  // 32768 equal (0.56 ms); the two-tile kernel wins at 65536 (2.07 against 2.15 ms)
  // and 131072 (7.95 against 8.41 ms: its units share each K/V block between two
  // tiles), and at L = 256 (11 against 13 us). Non-causal tiles carry equal work, so
  // there it wins only within one wave (2x8x512: 12.9 -> 11.9 us; 2x8x2048: 33.4
  // against 36.4 us).
  const bool alt_shape = !bf16 && d == 64;
  const long long alt_units = static_cast<long long>(B) * Hq * ((L + 127) / 128);
  const bool alt_auto = alt_shape && window_left < 0 && L >= 512 &&
                        (causal ? alt_units <= 8LL * info.sms : alt_units <= info.sms);
  const bool alt = alt_shape && (policy == ATTN_PATH_ALTERNATE || (policy == ATTN_PATH_AUTO && alt_auto));
  if (!alt && (policy == ATTN_PATH_TILES ||
               ((policy == ATTN_PATH_AUTO || policy == ATTN_PATH_ALTERNATE) && (few_units || tiles_win) &&
                Hq / Hkv <= 128)))
    return launch_square_as_kv(q, k, v, o, lse, B, L, Hq, Hkv, d, causal, window_left, -1, scale,
                               bf16, out_f32, workspace, stream, v16, vmax);
  CUtensorMap tm_q, tm_k, tm_v;
  if (!make_tensor_map(&tm_q, q, bf16, B, L, Hq, d, &why) ||
      !make_tensor_map(&tm_k, k, bf16, B, L, Hkv, d, &why) ||
      !(pv16 ? make_tensor_map(&tm_v, v16, false, B, L, Hkv, d, &why)
             : make_tensor_map(&tm_v, v, bf16, B, L, Hkv, d, &why)))
    return fail(ATTN_ERR_CUDA, why);

  ex19::LaunchArgs a = {};
  a.tm_q = &tm_q;
  a.tm_k = &tm_k;
  a.tm_v = &tm_v;
  ex19::FwdParams& p = a.p;
  p.o = o;
  p.lse = lse;
  p.status = static_cast<uint32_t*>(workspace);
  p.vmax = vmax;
  p.B = B;
  p.L = L;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.causal = causal;
  p.window_left = window_left;
  p.score_log2 = std::fabs(scale) * 1.4426950408889634f;
  p.negate_scores = scale < 0.f ? 1 : 0;
  p.units_per_bh = alt ? (L + 127) / 128 : (L + kUnitRows - 1) / kUnitRows;
  p.num_units = B * Hq * p.units_per_bh;
  p.wait_limit_ns = g_wait_limit_ns.load();
  a.grid = p.num_units < info.sms ? p.num_units : info.sms;
  a.stream = static_cast<cudaStream_t>(stream);
  // More two-tile units than CTAs: the CTAs take units from a counter in the
  // workspace (bytes 64..67, cleared here on the stream) instead of a static deal, so
  // that SMs that run faster take more of them (causal 4 heads d = 64 L = 131072:
  // 8.28 -> 7.93 ms; GQA d = 128 L = 16384 1.51 -> 1.48 ms; window 4096 3.67 -> 3.59
  // ms). The alternating mode keeps the static deal, which measured better for it
  // (L = 65536: 2.11 against 2.17 ms).
  if (!alt && p.num_units > a.grid) {
    uint32_t* counter = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + kSchedOffset);
    e = cudaMemsetAsync(counter, 0, sizeof(uint32_t), a.stream);
    if (e != cudaSuccess) return cuda_fail("clearing the unit counter", e);
    p.sched = counter;
  }

  if (alt) {
    e = ex19::launch_fwd_alt(out_f32, a);
  } else if (pv16) {
    e = ex19::launch_v_to_f16(v, v16, vmax, B, L, Hkv, d, a.stream);
    if (e != cudaSuccess) return cuda_fail("the fp16 copy of V", e);
    e = ex19::launch_fwd_pv16(d, out_f32, a);
  } else
    e = (d == 64) ? ex19::launch_fwd_d64(bf16, out_f32, a) : ex19::launch_fwd_d128(bf16, out_f32, a);
  if (e != cudaSuccess) return cuda_fail("kernel launch", e);
  return ATTN_OK;
}
}  // namespace ex19

extern "C" {

size_t attn_fwd_workspace_size(int B, int L, int Hq, int Hkv, int d, int causal, int window_left,
                               attn_dtype_t dtype) {
  if (check_shape(B, L, Hq, Hkv, d, causal, window_left) != ATTN_OK) return 0;
  if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return 0;
  return fwd_workspace_bytes(B, L, Hkv, d, dtype);
}

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int L, int Hq, int Hkv, int d, int causal, int window_left, float scale,
                       attn_dtype_t dtype, attn_out_t out_dtype, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return ex19::fwd_impl(q, k, v, o, lse, B, L, Hq, Hkv, d, causal, window_left, scale, dtype,
                        out_dtype, workspace, workspace_bytes, stream, 0);
}

attn_status_t attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int L, int Hq, int Hkv, int d, int window_left,
                              int window_right, float scale, attn_dtype_t dtype,
                              attn_out_t out_dtype, void* workspace, size_t workspace_bytes,
                              void* stream) {
  g_detail.clear();
  if (window_left < -1 || window_right < -1)
    return fail(ATTN_ERR_INVALID_ARG, "window_left and window_right must be >= -1");
  // the shape rules of attn_fwd, checked as a non-causal problem without a left window
  attn_status_t st = check_shape(B, L, Hq, Hkv, d, 0, -1);
  if (st != ATTN_OK) return st;
  if (Hq / Hkv > 128)
    return fail(ATTN_ERR_UNSUPPORTED, "at most 128 query heads may share one K/V head");
  if (!std::isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale must be finite");
  if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return fail(ATTN_ERR_INVALID_ARG, "bad dtype");
  if (out_dtype != ATTN_OUT_SAME && out_dtype != ATTN_OUT_FP32)
    return fail(ATTN_ERR_INVALID_ARG, "bad out_dtype");
  if (!q || !k || !v || !o) return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be non-null");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  if (!workspace) return fail(ATTN_ERR_WORKSPACE, "workspace must be non-null");
  if (!aligned(workspace, 16)) return fail(ATTN_ERR_WORKSPACE, "workspace must be 16-byte aligned");
  if (workspace_bytes < kWorkspaceBytes)
    return fail(ATTN_ERR_WORKSPACE, "workspace smaller than attn_fwd_workspace_size()");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  DeviceInfo info;
  if (!device_info(dev, &info, &e)) return cuda_fail("cudaDeviceGetAttribute", e);
  if (info.major != 10 || info.minor != 3)
    return fail(ATTN_ERR_UNSUPPORTED, "needs a compute capability 10.3 device (GB300), found " +
                                          std::to_string(info.major) + "." +
                                          std::to_string(info.minor));
  std::string why;
  const void* ptrs[6] = {q, k, v, o, workspace, lse};
  const char* names[6] = {"q", "k", "v", "o", "workspace", "lse"};
  for (int i = 0; i < 6; ++i)
    if (ptrs[i] && !is_device_ptr(ptrs[i], dev, &why, names[i]))
      return fail(ATTN_ERR_INVALID_ARG, why);
  return launch_square_as_kv(q, k, v, o, lse, B, L, Hq, Hkv, d, 0, window_left, window_right,
                             scale, dtype == ATTN_BF16, out_dtype == ATTN_OUT_FP32, workspace,
                             stream);
}

size_t attn_fwd_fp8_workspace_size(int B, int L, int Hq, int Hkv, int d, int causal,
                                   int window_left) {
  if (check_shape(B, L, Hq, Hkv, d, causal, window_left) != ATTN_OK) return 0;
  if (d != 64 || Hq / Hkv > 128) return 0;
  const size_t Lp = ((size_t)L + 15) / 16 * 16;
  return kWorkspaceBytes + (size_t)B * Hkv * 64 * Lp;
}

attn_status_t attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                           int L, int Hq, int Hkv, int d, int causal, int window_left,
                           float scale, attn_out_t out_dtype, void* workspace,
                           size_t workspace_bytes, void* stream) {
  g_detail.clear();
  attn_status_t st = check_shape(B, L, Hq, Hkv, d, causal, window_left);
  if (st != ATTN_OK) return st;
  if (d != 64) return fail(ATTN_ERR_UNSUPPORTED, "the float8 path has d = 64 only");
  if (Hq / Hkv > 128)
    return fail(ATTN_ERR_UNSUPPORTED, "at most 128 query heads may share one K/V head");
  if (!std::isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale must be finite");
  if (out_dtype != ATTN_OUT_SAME && out_dtype != ATTN_OUT_FP32)
    return fail(ATTN_ERR_INVALID_ARG, "bad out_dtype");
  if (!q || !k || !v || !o) return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be non-null");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  if (!workspace) return fail(ATTN_ERR_WORKSPACE, "workspace must be non-null");
  if (!aligned(workspace, 16)) return fail(ATTN_ERR_WORKSPACE, "workspace must be 16-byte aligned");
  const int Lp = (L + 15) / 16 * 16;
  if (workspace_bytes < kWorkspaceBytes + (size_t)B * Hkv * 64 * Lp)
    return fail(ATTN_ERR_WORKSPACE, "workspace smaller than attn_fwd_fp8_workspace_size()");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  DeviceInfo info;
  if (!device_info(dev, &info, &e)) return cuda_fail("cudaDeviceGetAttribute", e);
  if (info.major != 10 || info.minor != 3)
    return fail(ATTN_ERR_UNSUPPORTED, "needs a compute capability 10.3 device (GB300), found " +
                                          std::to_string(info.major) + "." +
                                          std::to_string(info.minor));
  std::string why;
  const void* ptrs[6] = {q, k, v, o, workspace, lse};
  const char* names[6] = {"q", "k", "v", "o", "workspace", "lse"};
  for (int i = 0; i < 6; ++i)
    if (ptrs[i] && !is_device_ptr(ptrs[i], dev, &why, names[i]))
      return fail(ATTN_ERR_INVALID_ARG, why);

  const KvPlan plan = kv_plan(B, L, L, Hq, Hkv, causal, window_left);
  uint8_t* vt = static_cast<uint8_t*>(workspace) + kWorkspaceBytes;
  CUtensorMap tm_q, tm_k, tm_vt;
  const cuuint64_t L64 = (cuuint64_t)L, Lp64 = (cuuint64_t)Lp;
  bool ok =
      make_tensor_map_u8(&tm_q, q, {64, (cuuint64_t)Hq, L64, (cuuint64_t)B},
                         {64, 64ull * Hq, 64ull * Hq * L64}, {64, (cuuint32_t)plan.group,
                                                             (cuuint32_t)plan.q_per_tile, 1},
                         CU_TENSOR_MAP_SWIZZLE_64B, &why) &&
      make_tensor_map_u8(&tm_k, k, {64, (cuuint64_t)Hkv, L64, (cuuint64_t)B},
                         {64, 64ull * Hkv, 64ull * Hkv * L64}, {64, 1, 128, 1},
                         CU_TENSOR_MAP_SWIZZLE_64B, &why) &&
      make_tensor_map_u8(&tm_vt, vt, {Lp64, 64, (cuuint64_t)Hkv, (cuuint64_t)B},
                         {Lp64, 64ull * Lp64, 64ull * Lp64 * Hkv}, {128, 64, 1, 1},
                         CU_TENSOR_MAP_SWIZZLE_128B, &why);
  if (!ok) return fail(ATTN_ERR_CUDA, why);

  ex19::Fp8LaunchArgs a = {};
  a.tm_q = &tm_q;
  a.tm_k = &tm_k;
  a.tm_vt = &tm_vt;
  ex19::KvParams& p = a.p;
  p.o = o;
  p.lse = lse;
  p.status = static_cast<uint32_t*>(workspace);
  p.B = B;
  p.Lq = L;
  p.Lk = L;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = plan.group;
  p.causal = causal;
  p.window_left = window_left;
  p.window_right = -1;
  p.score_log2 = std::fabs(scale) * 1.4426950408889634f;
  p.negate_scores = scale < 0.f ? 1 : 0;
  p.q_per_tile = plan.q_per_tile;
  p.row_tiles = plan.row_tiles;
  p.splits = 1;
  p.wait_limit_ns = g_wait_limit_ns.load();
  a.v = static_cast<const uint8_t*>(v);
  a.vt = vt;
  a.Lp = Lp;
  a.grid = plan.items;
  a.stream = static_cast<cudaStream_t>(stream);
  e = ex19::launch_fp8(out_dtype == ATTN_OUT_FP32, a);
  if (e != cudaSuccess) return cuda_fail("kernel launch", e);
  return ATTN_OK;
}

size_t attn_bwd_workspace_size(int B, int L, int Hq, int Hkv, int d, int causal,
                               int window_left) {
  if (check_shape(B, L, Hq, Hkv, d, causal, window_left) != ATTN_OK || Hq / Hkv > 128) return 0;
  const size_t Lpad = ((size_t)L + 127) / 128 * 128;
  return kWorkspaceBytes + 2 * (size_t)B * Hq * Lpad * 4;
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                       int L, int Hq, int Hkv, int d, int causal, int window_left, float scale,
                       attn_dtype_t dtype, attn_out_t out_dtype, void* workspace,
                       size_t workspace_bytes, void* stream) {
  g_detail.clear();
  attn_status_t st = check_shape(B, L, Hq, Hkv, d, causal, window_left);
  if (st != ATTN_OK) return st;
  if (Hq / Hkv > 128)
    return fail(ATTN_ERR_UNSUPPORTED, "at most 128 query heads may share one K/V head");
  if (!std::isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale must be finite");
  if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return fail(ATTN_ERR_INVALID_ARG, "bad dtype");
  if (out_dtype != ATTN_OUT_SAME && out_dtype != ATTN_OUT_FP32)
    return fail(ATTN_ERR_INVALID_ARG, "bad out_dtype");
  const void* in[6] = {q, k, v, o, dout, lse};
  void* out[3] = {dq, dk, dv};
  for (const void* x : in)
    if (!x) return fail(ATTN_ERR_INVALID_ARG, "q, k, v, o, lse and dout must be non-null");
  for (void* x : out)
    if (!x) return fail(ATTN_ERR_INVALID_ARG, "dq, dk and dv must be non-null");
  for (int i = 0; i < 5; ++i)
    if (!aligned(in[i], 16))
      return fail(ATTN_ERR_INVALID_ARG, "q, k, v, o and dout must be 16-byte aligned");
  if (!aligned(lse, 4)) return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  for (void* x : out)
    if (!aligned(x, 16)) return fail(ATTN_ERR_INVALID_ARG, "dq, dk and dv must be 16-byte aligned");
  if (!workspace) return fail(ATTN_ERR_WORKSPACE, "workspace must be non-null");
  if (!aligned(workspace, 16)) return fail(ATTN_ERR_WORKSPACE, "workspace must be 16-byte aligned");
  const int Lpad = (L + 127) / 128 * 128;
  if (workspace_bytes < kWorkspaceBytes + 2 * (size_t)B * Hq * Lpad * 4)
    return fail(ATTN_ERR_WORKSPACE, "workspace smaller than attn_bwd_workspace_size()");
  if ((long long)B * Hq * Lpad >= (1LL << 31))
    return fail(ATTN_ERR_INVALID_ARG, "B * Hq * L rounded up to 128 must be < 2^31");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  DeviceInfo info;
  if (!device_info(dev, &info, &e)) return cuda_fail("cudaDeviceGetAttribute", e);
  if (info.major != 10 || info.minor != 3)
    return fail(ATTN_ERR_UNSUPPORTED, "needs a compute capability 10.3 device (GB300), found " +
                                          std::to_string(info.major) + "." +
                                          std::to_string(info.minor));
  std::string why;
  const void* ptrs[10] = {q, k, v, o, dout, lse, dq, dk, dv, workspace};
  const char* names[10] = {"q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv", "workspace"};
  for (int i = 0; i < 10; ++i)
    if (!is_device_ptr(ptrs[i], dev, &why, names[i])) return fail(ATTN_ERR_INVALID_ARG, why);

  const bool bf16 = dtype == ATTN_BF16;
  const KvPlan plan = kv_plan(B, L, L, Hq, Hkv, causal, window_left);
  float* lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + kWorkspaceBytes);
  float* dsum = lse2 + (size_t)B * Hq * Lpad;
  CUtensorMap tm_qp, tm_dop, tm_q, tm_do, tm_k, tm_v, tm_lse2, tm_dsum;
  const bool maps_ok =
      make_tensor_map(&tm_qp, q, bf16, B, L, Hq, d, &why, plan.group, plan.q_per_tile) &&
      make_tensor_map(&tm_dop, dout, bf16, B, L, Hq, d, &why, plan.group, plan.q_per_tile) &&
      make_tensor_map(&tm_q, q, bf16, B, L, Hq, d, &why) &&
      make_tensor_map(&tm_do, dout, bf16, B, L, Hq, d, &why) &&
      make_tensor_map(&tm_k, k, bf16, B, L, Hkv, d, &why) &&
      make_tensor_map(&tm_v, v, bf16, B, L, Hkv, d, &why) &&
      make_tensor_map_f32_rows(&tm_lse2, lse2, B * Hq, Lpad, 128, &why) &&
      make_tensor_map_f32_rows(&tm_dsum, dsum, B * Hq, Lpad, 128, &why);
  if (!maps_ok) return fail(ATTN_ERR_CUDA, why);

  ex19::BwdLaunchArgs a = {};
  a.tm_qp = &tm_qp;
  a.tm_dop = &tm_dop;
  a.tm_q = &tm_q;
  a.tm_do = &tm_do;
  a.tm_k = &tm_k;
  a.tm_v = &tm_v;
  a.tm_lse2 = &tm_lse2;
  a.tm_dsum = &tm_dsum;
  ex19::bwd::BwdParams& p = a.p;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.lse2 = lse2;
  p.dsum = dsum;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.status = static_cast<uint32_t*>(workspace);
  p.B = B;
  p.L = L;
  p.Lpad = Lpad;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = plan.group;
  p.causal = causal;
  p.window_left = window_left;
  p.c2 = scale * 1.4426950408889634f;
  p.scale = scale;
  p.q_per_tile = plan.q_per_tile;
  p.row_tiles = plan.row_tiles;
  p.wait_limit_ns = g_wait_limit_ns.load();
  a.grid_dq = plan.items;
  a.grid_dkdv = B * Hkv * ((L + 127) / 128);
  a.stream = static_cast<cudaStream_t>(stream);
  e = ex19::launch_bwd(d, bf16, out_dtype == ATTN_OUT_FP32, a);
  if (e != cudaSuccess) return cuda_fail("kernel launch", e);
  return ATTN_OK;
}

int attn_fwd_kv_num_splits(int B, int Lq, int Lk, int Hq, int Hkv, int d, int causal,
                           int window_left) {
  if (check_kv_shape(B, Lq, Lk, Hq, Hkv, d, causal, window_left) != ATTN_OK) return 0;
  int sms = 0;
  if (current_sms(&sms) != 0) {
    fail(ATTN_ERR_CUDA, "no CUDA device");
    return 0;
  }
  return kv_auto_splits(kv_plan(B, Lq, Lk, Hq, Hkv, causal, window_left), sms);
}

size_t attn_fwd_kv_workspace_size(int B, int Lq, int Lk, int Hq, int Hkv, int d, int causal,
                                  int window_left, int num_splits) {
  if (check_kv_shape(B, Lq, Lk, Hq, Hkv, d, causal, window_left) != ATTN_OK) return 0;
  if (num_splits < 0 || num_splits > kKvMaxSplits) return 0;
  if (num_splits == 0) {
    num_splits = attn_fwd_kv_num_splits(B, Lq, Lk, Hq, Hkv, d, causal, window_left);
    if (num_splits == 0) return 0;
  }
  return kv_workspace_bytes(B, Lq, Hq, d, num_splits,
                            kv_plan(B, Lq, Lk, Hq, Hkv, causal, window_left).items);
}

attn_status_t attn_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int Lq, int Lk, int Hq, int Hkv, int d, int causal,
                          int window_left, float scale, attn_dtype_t dtype, attn_out_t out_dtype,
                          int num_splits, void* workspace, size_t workspace_bytes, void* stream) {
  return kv_run(q, k, v, o, lse, B, Lq, Lk, Hq, Hkv, d, causal, window_left, scale, dtype,
                out_dtype, num_splits, workspace, workspace_bytes, stream, nullptr);
}

attn_status_t attn_fwd_kv_paged(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, const int32_t* seq_lens, void* o,
                                float* lse, int B, int Lq, int Hq, int Hkv, int d, int page_size,
                                int num_pages, int max_pages_per_seq, int max_seq_len, int causal,
                                int window_left, float scale, attn_dtype_t dtype,
                                attn_out_t out_dtype, int num_splits, void* workspace,
                                size_t workspace_bytes, void* stream) {
  const PagedArgs pg = {block_table, seq_lens, page_size, num_pages, max_pages_per_seq};
  return kv_run(q, k_cache, v_cache, o, lse, B, Lq, max_seq_len, Hq, Hkv, d, causal, window_left,
                scale, dtype, out_dtype, num_splits, workspace, workspace_bytes, stream, &pg);
}

attn_status_t attn_fwd_sync_status(void* workspace, void* stream) {
  g_detail.clear();
  if (!workspace || !aligned(workspace, 16))
    return fail(ATTN_ERR_WORKSPACE, "workspace must be non-null and 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
  uint32_t word[4] = {0, 0, 0, 0};
  e = cudaMemcpyAsync(word, workspace, sizeof word, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail("reading the status word", e);
  if (word[0] == 0) return ATTN_OK;
  e = cudaMemsetAsync(workspace, 0, sizeof word, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail("clearing the status word", e);
  char buf[160];
  std::snprintf(buf, sizeof buf, "device status %u at site 0x%05x, CTA %u, unit %u", word[0],
                word[1], word[2], word[3]);
  attn_status_t code = (word[0] <= ATTN_ERR_TIMEOUT) ? static_cast<attn_status_t>(word[0])
                                                      : ATTN_ERR_CUDA;
  return fail(code, buf);
}

void attn_set_path_policy(int policy) {
  g_path_policy.store((policy == ATTN_PATH_SQUARE || policy == ATTN_PATH_TILES ||
                       policy == ATTN_PATH_ALTERNATE)
                          ? policy
                          : ATTN_PATH_AUTO);
}

int attn_get_path_policy(void) { return g_path_policy.load(); }

void attn_set_wait_limit_ns(uint64_t limit_ns) {
  g_wait_limit_ns.store(limit_ns ? (unsigned long long)limit_ns : kDefaultWaitLimitNs);
}

attn_status_t attn_debug_wait_probe(void* workspace, size_t workspace_bytes, uint64_t limit_ns,
                                    void* stream) {
  g_detail.clear();
  if (!workspace || !aligned(workspace, 16) || workspace_bytes < kWorkspaceBytes)
    return fail(ATTN_ERR_WORKSPACE, "workspace must be non-null, 16-byte aligned and large enough");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  DeviceInfo info;
  if (!device_info(dev, &info, &e)) return cuda_fail("cudaDeviceGetAttribute", e);
  if (info.major != 10 || info.minor != 3)
    return fail(ATTN_ERR_UNSUPPORTED, "needs a compute capability 10.3 device (GB300)");
  std::string why;
  if (!is_device_ptr(workspace, dev, &why, "workspace")) return fail(ATTN_ERR_INVALID_ARG, why);
  e = ex19::launch_wait_probe(static_cast<uint32_t*>(workspace), limit_ns,
                              static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("probe launch", e);
  return ATTN_OK;
}

int attn_debug_v16_exponent(uint32_t absmax_bits) { return ex19::v16_exponent(absmax_bits); }

attn_status_t attn_debug_exp2(const float* x, float* y_mufu, float* y_f16, int n, void* stream) {
  g_detail.clear();
  if (n < 0) return fail(ATTN_ERR_INVALID_ARG, "n must be >= 0");
  if (n == 0) return ATTN_OK;
  if (!x || !y_mufu) return fail(ATTN_ERR_INVALID_ARG, "pointers must be non-null");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  DeviceInfo info;
  if (!device_info(dev, &info, &e)) return cuda_fail("cudaDeviceGetAttribute", e);
  if (info.major != 10 || info.minor != 3)
    return fail(ATTN_ERR_UNSUPPORTED, "needs a compute capability 10.3 device (GB300)");
  std::string why;
  const void* ptrs[3] = {x, y_mufu, y_f16};
  const char* names[3] = {"x", "y_mufu", "y_f16"};
  for (int i = 0; i < 3; ++i)
    if (ptrs[i] && !is_device_ptr(ptrs[i], dev, &why, names[i]))
      return fail(ATTN_ERR_INVALID_ARG, why);
  e = ex19::launch_exp2_probe(x, y_mufu, y_f16, n, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("exp2 probe launch", e);
  return ATTN_OK;
}

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported";
    case ATTN_ERR_WORKSPACE: return "bad workspace";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

const char* attn_last_error_detail(void) { return g_detail.c_str(); }

int attn_abi_version(void) { return ATTN_ABI_VERSION; }

}  // extern "C"
