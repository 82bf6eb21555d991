// row_ops.cuh — per-thread operations on one row of a 128-key score block, and
// 16-bit packing helpers, shared by the attention kernels (one thread owns one
// query row; its 128 scores sit in registers after a TMEM load).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace ex19 {

// Maximum of a 128-value row: 8 independent chains (16 values each, 3-input
// maxima), then a tree.
__device__ __forceinline__ float row_max128(const float (&s)[128]) {
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a = max3f(s[i], s[8 + i], s[16 + i]);
#pragma unroll
    for (int k = 24; k < 120; k += 16) a = max3f(a, s[k + i], s[k + 8 + i]);  // 24 .. 112
    m[i] = fmaxf(a, s[120 + i]);
  }
  return max3f(max3f(m[0], m[1], m[2]), max3f(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// Minimum of a 128-value row (used when the scale is negative).
__device__ __forceinline__ float row_min128(const float (&s)[128]) {
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a = s[i];
#pragma unroll
    for (int k = 8; k < 128; k += 8) a = fminf(a, s[k + i]);
    m[i] = a;
  }
  return fminf(fminf(fminf(m[0], m[1]), fminf(m[2], m[3])), fminf(fminf(m[4], m[5]), fminf(m[6], m[7])));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float low_as_float(uint32_t packed, bool bf16) {
  if (bf16) return __uint_as_float(packed << 16);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(packed & 0xFFFFu)));
}

__device__ __forceinline__ float high_as_float(uint32_t packed, bool bf16) {
  if (bf16) return __uint_as_float(packed & 0xFFFF0000u);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(packed >> 16)));
}

}  // namespace ex19
