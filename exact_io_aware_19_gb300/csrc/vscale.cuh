// vscale.cuh — the per-head power-of-two scale of the fp16 copy of a bfloat16 V.
//
// With bfloat16 inputs the attention weights P enter the P·V product as fp16 (11
// significant bits) instead of bf16 (8), so that one product per key block suffices
// (a bf16 P needs a hi + lo pair of products to stay within the output tolerance).
// The product's two operands must share one type, so V is re-encoded once per call:
// V16 = fp16(V · 2^e) with one exponent e per (batch, K/V head), chosen from the
// largest finite |v| of that head so that it lands in [2^14, 2^15) (fp16's largest
// finite value is 65504 < 2^16). A bfloat16 value has 8 significant bits and fp16
// 11, so every scaled value at or above 2^-17 (fp16's subnormal spacing 2^-24 times
// 2^7) is represented exactly; smaller ones, below 2^-31 of the head's largest |v|,
// are rounded to the nearest multiple of 2^-24. The output undoes the scale:
// O = (Σ P · V16) · 2^-e / l, a power-of-two multiply, exact in fp32.
//
// Infinities and NaNs are left out of the maximum; they convert to themselves.
#pragma once
#include <cstdint>

namespace ex19 {

// The exponent e for a head whose largest finite |v| has bfloat16 bits `absmax`
// (sign clear; 0 for an all-zero head). Normal maxima m = 1.f × 2^(E - 127) give
// e = 14 - (E - 127); subnormal maxima, and heads below 2^-112, take e = 126, the
// largest exponent whose 2^e and 2^-e are both normal floats.
__host__ __device__ __forceinline__ int v16_exponent(uint32_t absmax) {
  if (absmax == 0u) return 0;
  const int E = static_cast<int>((absmax >> 7) & 0xFFu);  // bf16 exponent field
  if (E == 0) return 126;
  const int e = 141 - E;
  return e > 126 ? 126 : e;
}

// 2^k for |k| <= 126, exactly.
__host__ __device__ __forceinline__ float exp2_int(int k) {
  const uint32_t bits = static_cast<uint32_t>(k + 127) << 23;
  float f;
  __builtin_memcpy(&f, &bits, 4);
  return f;
}

}  // namespace ex19
