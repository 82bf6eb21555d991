// attn_bwd_params.h — parameter block of the backward pass, shared by the host
// launcher and the kernels.
#pragma once
#include <cstdint>

namespace ex19 {
namespace bwd {

struct BwdParams {
  const void* o;       // [B, L, Hq, D] forward output (input dtype)
  const void* dout;    // [B, L, Hq, D] upstream gradient
  const float* lse;    // [B, Hq, L] forward log-sum-exp (natural log)
  float* lse2;         // workspace [B * Hq, Lpad]: LSE in base 2 (+inf past L)
  float* dsum;         // workspace [B * Hq, Lpad]: D (0 past L)
  void* dq;            // [B, L, Hq, D] (input dtype or float32)
  void* dk;            // [B, L, Hkv, D]
  void* dv;            // [B, L, Hkv, D]
  uint32_t* status;
  int B, L, Lpad, Hq, Hkv, group;
  int causal, window_left;
  float c2;            // scale * log2(e) (signed)
  float scale;
  int q_per_tile, row_tiles;  // dQ kernel: query positions per packed 128-row tile
  unsigned long long wait_limit_ns;
};

}  // namespace bwd
}  // namespace ex19
