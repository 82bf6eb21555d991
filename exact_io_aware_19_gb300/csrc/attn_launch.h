// attn_launch.h — host-side entry points of the per-head-dim kernel instantiations.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_bwd_params.h"
#include "attn_kv_params.h"
#include "attn_params.h"

namespace ex19 {

struct LaunchArgs {
  const CUtensorMap* tm_q;
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  FwdParams p;
  int grid;
  cudaStream_t stream;
};

struct KvLaunchArgs {
  const CUtensorMap* tm_q;
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  KvParams p;
  int grid;  // B * Hkv * row_tiles * splits
  cudaStream_t stream;
};

struct Fp8LaunchArgs {
  const CUtensorMap* tm_q;
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_vt;  // over vt
  KvParams p;                // Lq = Lk = L, splits = 1
  const uint8_t* v;          // [B, L, Hkv, 64] e4m3
  uint8_t* vt;               // [B, Hkv, 64, Lp] e4m3, in the workspace
  int Lp;                    // L rounded up to 16
  int grid;                  // B * Hkv * row_tiles
  cudaStream_t stream;
};

struct BwdLaunchArgs {
  const CUtensorMap* tm_qp;   // Q, packed 128-row tiles (dQ kernel)
  const CUtensorMap* tm_dop;  // dO, packed likewise
  const CUtensorMap* tm_q;    // Q, one head per 128-row tile (dK / dV kernel)
  const CUtensorMap* tm_do;   // dO, likewise
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  const CUtensorMap* tm_lse2;  // [B * Hq, Lpad] float32, boxes of 128
  const CUtensorMap* tm_dsum;
  bwd::BwdParams p;
  int grid_dq, grid_dkdv;
  cudaStream_t stream;
};

// Each returns the CUDA error of configuring / enqueuing the kernel.
cudaError_t launch_fwd_d64(bool bf16, bool out_f32, const LaunchArgs& a);
cudaError_t launch_fwd_d128(bool bf16, bool out_f32, const LaunchArgs& a);
// The alternating mode (fp16, d = 64): one 128-row tile per work unit, both
// pipelines on alternate key blocks (a.p.units_per_bh = ceil(L / 128)).
cudaError_t launch_fwd_alt(bool out_f32, const LaunchArgs& a);
// bfloat16 inputs with the fp16 copy of V (a.tm_v over it, a.p.vmax set).
cudaError_t launch_fwd_pv16(int d, bool out_f32, const LaunchArgs& a);
// The fp16 copy of a bfloat16 V [B, L, Hkv, d] with one power-of-two scale per
// (batch, K/V head): clears vmax [B * Hkv], writes the heads' largest finite |v|
// there, then v16 (the same layout as v). Three operations on `stream`.
cudaError_t launch_v_to_f16(const void* v, void* v16, uint32_t* vmax, int B, int L, int Hkv,
                            int d, cudaStream_t stream);
// The decode-shaped forward (and, when p.splits > 1, its merge kernel).
cudaError_t launch_kv(int d, bool bf16, bool out_f32, const KvLaunchArgs& a);
// The one-tile kernel for attn_fwd on bfloat16 inputs with the fp16 copy of V (one
// key split; a.tm_v over the copy, a.p.vmax set).
cudaError_t launch_kv_pv16(int d, bool out_f32, const KvLaunchArgs& a);
// Work items of at most 32 query rows (q_per_tile * group) run the keys-on-lanes
// kernel (attn_kv_keys_kernel.cuh), one CTA per SM.
inline bool kv_keys_shape(int q_per_tile, int group) { return q_per_tile * group <= 32; }
cudaError_t launch_kv_keys(int d, bool bf16, bool paged, bool out_f32, const KvLaunchArgs& a);
// The merge of a.p.splits > 1 partial results into O and LSE.
cudaError_t launch_kv_merge(int d, bool bf16, bool out_f32, const KvLaunchArgs& a);
// The same over a paged K/V cache (a.p.block_table, seq_lens, page_size, ... set).
cudaError_t launch_kv_paged(int d, bool bf16, bool out_f32, const KvLaunchArgs& a);
// The float8 forward: the V transpose, then the attention kernel.
cudaError_t launch_fp8(bool out_f32, const Fp8LaunchArgs& a);
// The backward pass: the D / LSE2 pass, the dQ kernel and the dK / dV kernel.
cudaError_t launch_bwd(int d, bool bf16, bool out_f32, const BwdLaunchArgs& a);
cudaError_t launch_wait_probe(uint32_t* status, unsigned long long limit_ns, cudaStream_t stream);
cudaError_t launch_exp2_probe(const float* x, float* y_mufu, float* y_f16, int n,
                              cudaStream_t stream);

}  // namespace ex19
