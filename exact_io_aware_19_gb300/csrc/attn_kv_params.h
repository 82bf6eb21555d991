// attn_kv_params.h — parameter block of the decode-shaped (split-KV) forward, shared
// by the host launcher and the kernels.
#pragma once
#include <cstdint>

namespace ex19 {

struct KvParams {
  void* o;              // [B, Lq, Hq, D], input dtype or float32
  float* lse;           // [B, Hq, Lq] or null
  uint32_t* status;     // 4 x u32 status word in the workspace
  float* o_part;        // [splits, B*Hq*Lq, D] float32 partial outputs (splits > 1), else null
  float* lse_part;      // [splits, B*Hq*Lq] partial log2-sum-exp (splits > 1), else null
  const uint32_t* vmax; // [B, Hkv] largest finite |v| (bf16 bits) of the fp16 copy of V, or null
  // Merge tickets of the keys-on-lanes kernel (splits > 1): one 64-bit word per work
  // item, (call tag << 9) | CTAs of the item that have stored their partial result.
  unsigned long long* tickets;
  unsigned long long ticket_base;  // this call's tag << 9 (low 9 bits zero)
  int B, Lq, Lk, Hq, Hkv;
  int group;            // Hq / Hkv: query heads that read one K/V head
  int causal;           // 0 / 1
  int window_left;      // -1 or >= 0
  int window_right;     // -1 or >= 0: keys j <= position + window_right (causal acts as 0)
  float score_log2;     // |scale| * log2(e)
  int negate_scores;    // 1 when scale < 0
  int q_per_tile;       // query positions per 128-row tile (each with all `group` heads)
  int row_tiles;        // ceil(Lq / q_per_tile)
  int splits;           // key-range splits per (batch, K/V head, row tile)
  unsigned long long wait_limit_ns;
  // Paged K/V cache (paged kernels only): k, v are [num_pages, page_size, Hkv, D];
  // sequence b's key t sits at row t % page_size of page block_table[b * max_pages +
  // t / page_size]; its length is seq_lens[b] (Lq <= seq_lens[b] <= Lk, the maximum).
  const int* block_table;
  const int* seq_lens;
  int page_size;        // divides 128
  int max_pages;        // row stride of block_table
  int num_pages;
};

}  // namespace ex19
