// attn_params.h — plain parameter block shared by the host launcher and the kernel.
#pragma once
#include <cstdint>

namespace ex19 {

struct FwdParams {
  void* o;              // [B, L, Hq, D], input dtype or float32
  float* lse;           // [B, Hq, L] or null
  uint32_t* status;     // 4 x u32 status word in the workspace, or null
  const uint32_t* vmax; // [B, Hkv] largest finite |v| (bf16 bits) of the fp16 copy of V, or null
  uint32_t* sched;      // dynamic scheduling: a zeroed counter of unit ranks taken, or null (static)
  int B, L, Hq, Hkv;
  int causal;           // 0 / 1
  int window_left;      // -1 or >= 0
  float score_log2;     // |scale| * log2(e): x = score_log2 * (±q·k)
  int negate_scores;    // 1 when scale < 0 (scores are negated, score_log2 stays >= 0)
  int units_per_bh;     // ceil(L / 256): 256-row work units per (batch, head)
  int num_units;        // B * Hq * units_per_bh
  unsigned long long wait_limit_ns;
};

}  // namespace ex19
