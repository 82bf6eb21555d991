// attn_vconv.cu — the fp16 copy of a bfloat16 V with a per-head power-of-two scale
// (the exponent rule and its exactness are stated in vscale.cuh).
//
// Two HBM-bound passes over V [B, L, Hkv, d]: the largest finite |v| of every
// (batch, K/V head), then the scaled conversion. Both read V as rows of Hkv·d
// elements in 16-byte pieces (8 values of one head, since d is a multiple of 8):
// consecutive threads take consecutive pieces of a row, so each warp reads 512
// contiguous bytes, and each thread keeps four loads in flight.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_launch.h"
#include "vscale.cuh"

namespace ex19 {
namespace {

constexpr int kRowsPerCta = 32;  // rows of V per CTA
constexpr int kUnroll = 4;       // 16-byte loads in flight per thread

// Both kernels run on the grid (B * ceil(L / kRowsPerCta), ceil(pieces / blockDim.x)),
// pieces = Hkv·d/8 16-byte pieces per row: a CTA takes kRowsPerCta rows of one batch
// entry, a thread one piece column of them, so its (batch, head) is fixed.
struct PieceCol {
  int b, r0, r1, c;
  bool live;
};

__device__ __forceinline__ PieceCol piece_col(int L, int pieces) {
  PieceCol pc;
  const int row_blocks = (L + kRowsPerCta - 1) / kRowsPerCta;
  pc.b = blockIdx.x / row_blocks;
  pc.r0 = (blockIdx.x % row_blocks) * kRowsPerCta;
  pc.r1 = min(L, pc.r0 + kRowsPerCta);
  pc.c = blockIdx.y * blockDim.x + threadIdx.x;
  pc.live = pc.c < pieces;
  return pc;
}

__device__ __forceinline__ uint32_t abs_max8(const uint4 w) {
  uint32_t m = 0;
  const uint32_t parts[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = parts[i] & 0x7FFFu, hi = (parts[i] >> 16) & 0x7FFFu;
    // bit patterns of |v| order like the values; 0x7F80 and above are inf / NaN
    if (lo < 0x7F80u) m = max(m, lo);
    if (hi < 0x7F80u) m = max(m, hi);
  }
  return m;
}

// vmax[b * Hkv + g] = max over the head's finite |v| (bf16 bits), by atomicMax on a
// zeroed array. The pieces of one head are d/8 consecutive threads, aligned within
// the warp (d/8 divides 32 and blockDim.x is a multiple of 32), reduced by shuffles.
__global__ void __launch_bounds__(256) v_absmax_kernel(const uint4* __restrict__ v,
                                                       uint32_t* __restrict__ vmax, int L,
                                                       int Hkv, int d) {
  const int pieces = Hkv * d / 8;
  const PieceCol pc = piece_col(L, pieces);
  uint32_t m = 0;
  if (pc.live) {
    const uint4* base = v + static_cast<size_t>(pc.b) * L * pieces + pc.c;
    int r = pc.r0;
    for (; r + kUnroll <= pc.r1; r += kUnroll) {
      uint4 w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) w[u] = __ldg(base + static_cast<size_t>(r + u) * pieces);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) m = max(m, abs_max8(w[u]));
    }
    for (; r < pc.r1; ++r) m = max(m, abs_max8(__ldg(base + static_cast<size_t>(r) * pieces)));
  }
  const int group = d / 8;  // 8 or 16 lanes per head
  for (int off = group >> 1; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (pc.live && (pc.c % group) == 0 && m != 0u) atomicMax(vmax + pc.b * Hkv + pc.c / group, m);
}

__device__ __forceinline__ uint32_t to_f16x2_scaled(uint32_t bf2, float s) {
  const float lo = __uint_as_float(bf2 << 16) * s;
  const float hi = __uint_as_float(bf2 & 0xFFFF0000u) * s;
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint4 to_f16x8_scaled(const uint4 w, float s) {
  uint4 o;
  o.x = to_f16x2_scaled(w.x, s);
  o.y = to_f16x2_scaled(w.y, s);
  o.z = to_f16x2_scaled(w.z, s);
  o.w = to_f16x2_scaled(w.w, s);
  return o;
}

// v16 = fp16(v · 2^e(b, g)), the same layout as v.
__global__ void __launch_bounds__(256) v_to_f16_kernel(const uint4* __restrict__ v,
                                                       uint4* __restrict__ v16,
                                                       const uint32_t* __restrict__ vmax, int L,
                                                       int Hkv, int d) {
  const int pieces = Hkv * d / 8;
  const PieceCol pc = piece_col(L, pieces);
  if (!pc.live) return;
  const float s = exp2_int(v16_exponent(__ldg(vmax + pc.b * Hkv + pc.c / (d / 8))));
  const size_t base = static_cast<size_t>(pc.b) * L * pieces + pc.c;
  int r = pc.r0;
  for (; r + kUnroll <= pc.r1; r += kUnroll) {
    uint4 w[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) w[u] = __ldg(v + base + static_cast<size_t>(r + u) * pieces);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v16[base + static_cast<size_t>(r + u) * pieces] = to_f16x8_scaled(w[u], s);
  }
  for (; r < pc.r1; ++r)
    v16[base + static_cast<size_t>(r) * pieces] = to_f16x8_scaled(__ldg(v + base + static_cast<size_t>(r) * pieces), s);
}

}  // namespace

cudaError_t launch_v_to_f16(const void* v, void* v16, uint32_t* vmax, int B, int L, int Hkv,
                            int d, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(vmax, 0, static_cast<size_t>(B) * Hkv * 4, stream);
  if (e != cudaSuccess) return e;
  const int pieces = Hkv * d / 8;
  const int threads = pieces >= 256 ? 256 : ((pieces + 31) / 32) * 32;
  const long long row_blocks = (L + kRowsPerCta - 1) / kRowsPerCta;
  const long long gx = static_cast<long long>(B) * row_blocks;
  const long long gy = (pieces + threads - 1) / threads;
  if (gx >= (1LL << 31) || gy > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  v_absmax_kernel<<<grid, threads, 0, stream>>>(static_cast<const uint4*>(v), vmax, L, Hkv, d);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  v_to_f16_kernel<<<grid, threads, 0, stream>>>(static_cast<const uint4*>(v), static_cast<uint4*>(v16),
                                                vmax, L, Hkv, d);
  return cudaGetLastError();
}

}  // namespace ex19
