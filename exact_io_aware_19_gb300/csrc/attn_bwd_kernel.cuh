// attn_bwd_kernel.cuh — gradients of exact attention (backward pass) for sm_103a.
//
// What it computes: for an upstream gradient dO of O, the gradients of the square
// problem's definition (the backward pass that the spec page "compare Hyena vs
// FlashAttention at 128k", stage 5, lists as not measured):
//   P_ij  = 2^(s_ij · c − LSE2_i) on the visible keys (c = scale · log2 e, LSE2 the
//           forward's log-sum-exp in base 2), D_i = Σ_c dO_ic O_ic,
//   dP_ij = dO_i · v_j,  dS_ij = P_ij (dP_ij − D_i),
//   dQ_i  = scale Σ_j dS_ij k_j,  dK_j = scale Σ_i dS_ij q_i,  dV_j = Σ_i P_ij dO_i,
// with dK and dV summed over the query heads of each K/V head. Nothing of size
// L x L is stored: like the forward, both kernels recompute S block by block.
//
// GB300 mapping: three kernels, each with the forward's warp roles (4 elementwise
// warps, one TMA producer warp, one MMA warp; every wait bounded):
//   * attn_bwd_prep: D and LSE2 per row into the workspace.
//   * attn_bwd_dq_kernel (query-stationary, one CTA per 128-row tile packed as in
//     the one-tile forward): per key block, S = Q Kᵀ and dP = dO Vᵀ (SS MMAs into
//     TMEM), dS written as 16-bit over the dP columns, then dQ += dS · K (A = dS from
//     TMEM, B = K MN-major in shared memory).
//   * attn_bwd_dkdv_kernel (key-stationary, one CTA per (batch, K/V head, 128-key
//     tile)): per (query head of the group, query block), Sᵀ = K Qᵀ and dPᵀ = V dOᵀ,
//     Pᵀ and dSᵀ written over them, then dV += Pᵀ · dO and dK += dSᵀ · Q.
// The MMA issue is serial per block: S and dP, then the elementwise pass, then the
// accumulating MMAs (TMEM holds one block's S and dP).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <type_traits>

#include "attn_bwd_params.h"
#include "row_ops.cuh"
#include "sm103_ptx.cuh"
#include "tmem_io.cuh"

namespace ex19 {
namespace bwd {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kThreads = 192;  // 4 elementwise warps + producer warp + MMA warp
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;

enum : uint32_t {
  kSiteProd = 0xE0001, kSiteMma = 0xE0002, kSiteEw = 0xE0003, kSiteDrain = 0xE0004,
};



// ------------------------------------------------------------------------ D, LSE2
// One warp per (b, h, i) row of [B, Hq, Lpad]: D = Σ dO·O, LSE2 = LSE · log2 e.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_prep(const BwdParams p) {
  const size_t row = static_cast<size_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<size_t>(p.B) * p.Hq * p.Lpad) return;
  const int i = static_cast<int>(row % p.Lpad);
  const size_t bh = row / p.Lpad;
  const int h = static_cast<int>(bh % p.Hq), b = static_cast<int>(bh / p.Hq);
  float dsum = 0.f, lse2 = INFINITY;
  if (i < p.L) {
    const size_t off = ((static_cast<size_t>(b) * p.L + i) * p.Hq + h) * D;
    const uint16_t* o = static_cast<const uint16_t*>(p.o) + off;
    const uint16_t* g = static_cast<const uint16_t*>(p.dout) + off;
    for (int c = lane; c < D; c += 32) {
      const uint32_t ov = o[c], gv = g[c];
      dsum += low_as_float(ov, BF16) * low_as_float(gv, BF16);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, s);
    const float l = p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.L + i];
    lse2 = l * 1.4426950408889634f;  // -inf stays -inf (a row with no visible key)
  }
  if (lane == 0) {
    p.dsum[row] = dsum;
    p.lse2[row] = lse2;
  }
}

// Geometry shared by both kernels: a resident pair of 128-row tiles and a ring of
// streamed tiles (pairs), all 128 rows x D 16-bit values in 128-byte swizzle boxes.
template <int D>
struct BwdGeometry {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = kBM * 128;
  static constexpr int kTileBytes = kBM * D * 2;
  static constexpr int kSlots = (D == 64) ? 8 : 4;  // streamed tiles
  static constexpr int kOffRes = 0;                 // 2 resident tiles
  static constexpr int kOffRing = 2 * kTileBytes;
  static constexpr int kOffVec = kOffRing + kSlots * kTileBytes;  // dK/dV kernel: LSE2, D rows
  static constexpr int kVecBytes = 2 * kBN * 4;                   // per stage
  static constexpr int kOffBar = kOffVec + (kSlots / 2) * kVecBytes;
  // barriers: full[S], empty[S], res_full, s_full, p_full, acc_done, drain
  static constexpr int kNumBars = 2 * kSlots + 5;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemUsed = kOffMisc + 16;
  static constexpr int kSmemBytes = kSmemUsed + 1024;
};

// The 16-bit pair of a fp32 pair in the input dtype.
__device__ __forceinline__ uint32_t pack_in(float a, float b, bool bf16) { return pack2(a, b, bf16); }

// Common preamble of both kernels: barriers, TMEM, wait control.
#define EX19_BWD_PREAMBLE()                                                                    \
  using G = BwdGeometry<D>;                                                                    \
  constexpr int S = G::kSlots;                                                                 \
  extern __shared__ uint8_t smem_raw[];                                                        \
  uint8_t* smem = reinterpret_cast<uint8_t*>(                                                  \
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));         \
  const uint32_t sbase = smem_u32(smem);                                                       \
  const uint32_t sRes = sbase + G::kOffRes;                                                    \
  const uint32_t sRing = sbase + G::kOffRing;                                                  \
  const uint32_t sVec = sbase + G::kOffVec;                                                    \
  const uint32_t bars = sbase + G::kOffBar;                                                    \
  auto bar_full = [&](uint32_t s) { return bars + 8u * s; };                                   \
  auto bar_empty = [&](uint32_t s) { return bars + 8u * (S + s); };                            \
  const uint32_t bar_res = bars + 8u * (2 * S);                                                \
  const uint32_t bar_s_full = bars + 8u * (2 * S + 1);                                         \
  const uint32_t bar_p_full = bars + 8u * (2 * S + 2);                                         \
  const uint32_t bar_acc_done = bars + 8u * (2 * S + 3);                                       \
  const uint32_t bar_drain = bars + 8u * (2 * S + 4);                                          \
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::kOffMisc);                       \
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + G::kOffMisc + 4); \
  const int warp = threadIdx.x >> 5;                                                           \
  const int lane = threadIdx.x & 31;                                                           \
  if (threadIdx.x == 0) {                                                                      \
    for (int s = 0; s < S; ++s) {                                                              \
      mbar_init(bar_full(s), 1);                                                               \
      mbar_init(bar_empty(s), 1);                                                              \
    }                                                                                          \
    mbar_init(bar_res, 1);                                                                     \
    mbar_init(bar_s_full, 1);                                                                  \
    mbar_init(bar_p_full, kBM);                                                                \
    mbar_init(bar_acc_done, 1);                                                                \
    mbar_init(bar_drain, 1);                                                                   \
    *abort_flag = 0u;                                                                          \
    fence_mbar_init();                                                                         \
  }                                                                                            \
  if (warp == kMmaWarp) {                                                                      \
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);                                                \
    tmem_relinquish();                                                                         \
  }                                                                                            \
  tc_fence_before();                                                                           \
  __syncthreads();                                                                             \
  tc_fence_after();                                                                            \
  const uint32_t tmem_base = *tmem_slot;                                                       \
  WaitCtl wc;                                                                                  \
  wc.abort_flag = abort_flag;                                                                  \
  wc.status = p.status;                                                                        \
  wc.limit_ns = p.wait_limit_ns;                                                               \
  wc.unit = blockIdx.x;

#define EX19_BWD_TEARDOWN()            \
  tc_fence_before();                   \
  __syncthreads();                     \
  tc_fence_after();                    \
  if (warp == kMmaWarp) {              \
    __syncwarp();                      \
    tmem_dealloc(tmem_base, kTmemCols); \
  }

// Elementwise pass of one block, shared by both kernels. The thread's row of the
// first operand block X (S or Sᵀ, fp32, columns [x0, x0+128)) and of dX (dP or dPᵀ,
// at dx0) become, 64 columns at a time: W = 2^(X·c − lse2[col]) (0 outside
// [vis_lo, vis_hi)), dS = W (dX − dsum[col]); W (if kStoreW) and dS are written as
// 16-bit pairs over the already-read first 64 columns of X and dX. lse2 / dsum per
// column come from `vec_col(c)` (dK/dV kernel) or are the row's own values.
template <bool BF16, bool kStoreW, typename VecFn>
__device__ __forceinline__ void elementwise_block(uint32_t tX, uint32_t tdX, float c2, int vis_lo,
                                                  int vis_hi, bool masked, VecFn vec_col) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t xs[64], dxs[64];
    tmem_ld_x64(tX + 64 * half, xs);
    tmem_ld_x64(tdX + 64 * half, dxs);
    uint32_t wpk[32], dspk[32];
#pragma unroll
    for (int c = 0; c < 64; c += 2) {
      const int cc = 64 * half + c;
      float l0, d0, l1, d1;
      vec_col(cc, l0, d0);
      vec_col(cc + 1, l1, d1);
      float w0 = ex2_approx(__uint_as_float(xs[c]) * c2 - l0);
      float w1 = ex2_approx(__uint_as_float(xs[c + 1]) * c2 - l1);
      if (masked) {
        w0 = (cc >= vis_lo && cc < vis_hi) ? w0 : 0.f;
        w1 = (cc + 1 >= vis_lo && cc + 1 < vis_hi) ? w1 : 0.f;
      }
      const float s0 = w0 * (__uint_as_float(dxs[c]) - d0);
      const float s1 = w1 * (__uint_as_float(dxs[c + 1]) - d1);
      wpk[c >> 1] = pack_in(w0, w1, BF16);
      dspk[c >> 1] = pack_in(s0, s1, BF16);
    }
    // 16-bit results over columns this thread has read: half h goes to 32h .. 32h+31
    if constexpr (kStoreW) {
      tmem_st_x32(tX + 32 * half, wpk);
    }
    tmem_st_x32(tdX + 32 * half, dspk);
  }
}

// ------------------------------------------------------------------------- dQ
template <int D, bool BF16, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const BwdParams p) {
  EX19_BWD_PREAMBLE()
  // item: (batch, K/V head, packed row tile)
  int x = blockIdx.x;
  const int rt = x % p.row_tiles;
  x /= p.row_tiles;
  const int g = x % p.Hkv, b = x / p.Hkv;
  const int i0 = rt * p.q_per_tile, i1 = min(p.L, i0 + p.q_per_tile);
  const int nblk = (p.L + kBN - 1) / kBN;
  const int blk_hi = p.causal ? (i1 - 1) / kBN + 1 : nblk;
  const int blk_lo = (p.window_left >= 0) ? max(0, i0 - p.window_left) / kBN : 0;
  const int nblocks = max(0, blk_hi - blk_lo);
  // TMEM: S [0,128), dP [128,256), dQ [256, 256 + D)
  const uint32_t kColS = 0, kColDP = 128, kColDQ = 256;

  if (warp == kProducerWarp) {
    if (lane == 0 && nblocks > 0) {
      const uint32_t qbytes = G::kChunks * 128u * p.group * p.q_per_tile;
      mbar_arrive_expect_tx(bar_res, 2 * qbytes);
      for (int c = 0; c < G::kChunks; ++c) {
        tma_load_4d(sRes + c * G::kChunkBytes, &tm_q, bar_res, c * 64, g * p.group, i0, b);
        tma_load_4d(sRes + G::kTileBytes + c * G::kChunkBytes, &tm_do, bar_res, c * 64,
                    g * p.group, i0, b);
      }
      uint32_t n = 0;
      bool ok = true;
      for (int j = blk_lo; ok && j < blk_hi; ++j) {
        for (int kv = 0; kv < 2; ++kv) {
          const uint32_t slot = n % S;
          ok = mbar_wait_bounded(bar_empty(slot), ((n / S) & 1u) ^ 1u, wc, kSiteProd);
          if (!ok) break;
          mbar_arrive_expect_tx(bar_full(slot), G::kTileBytes);
          for (int c = 0; c < G::kChunks; ++c)
            tma_load_4d(sRing + slot * G::kTileBytes + c * G::kChunkBytes, kv ? &tm_v : &tm_k,
                        bar_full(slot), c * 64, g, j * kBN, b);
          ++n;
        }
      }
      if (!ok) {
        for (uint32_t back = 1; back <= S && back <= n; ++back) {
          const uint32_t m = n - back;
          mbar_wait_drain(bar_full(m % S), (m / S) & 1u, wc, kSiteDrain);
        }
        mbar_wait_drain(bar_res, 0, wc, kSiteDrain);
      }
    }
  } else if (warp == kMmaWarp) {
    if (nblocks > 0) {
      constexpr uint32_t idesc_s = idesc_f16_f32acc(BF16, kBM, kBN, false);
      constexpr uint32_t idesc_q = idesc_f16_f32acc(BF16, kBM, D, true);
      const uint64_t dq_ = sdesc_sw128(sRes, 16, 1024);                   // Q, K-major
      const uint64_t ddo = sdesc_sw128(sRes + G::kTileBytes, 16, 1024);   // dO, K-major
      const uint64_t dkv = sdesc_sw128(sRing, 16, 1024);                  // K / V, K-major
      const uint64_t dkmn = sdesc_sw128(sRing, G::kChunkBytes, 1024);     // K, MN-major
      bool ok = mbar_wait_warp(bar_res, 0, wc, kSiteMma);
      for (int jj = 0; ok && jj < nblocks; ++jj) {
        const uint32_t kidx = 2u * jj, vidx = kidx + 1u;
        ok = mbar_wait_warp(bar_full(kidx % S), (kidx / S) & 1u, wc, kSiteMma) &&
             mbar_wait_warp(bar_full(vidx % S), (vidx / S) & 1u, wc, kSiteMma);
        if (!ok) break;
        tc_fence_after();
        const uint64_t kslot = ((kidx % S) * G::kTileBytes) >> 4;
        const uint64_t vslot = ((vidx % S) * G::kTileBytes) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * G::kChunkBytes + (kk & 3) * 32) >> 4;
          mma_ss_elect(tmem_base + kColS, dq_ + off, dkv + kslot + off, idesc_s, kk > 0);
          mma_ss_elect(tmem_base + kColDP, ddo + off, dkv + vslot + off, idesc_s, kk > 0);
        }
        mma_commit_elect(bar_s_full);
        mma_commit_elect(bar_empty(vidx % S));  // V_j is only read by dP
        ok = mbar_wait_warp(bar_p_full, jj & 1u, wc, kSiteMma);
        if (!ok) break;
        tc_fence_after();
        // dQ += dS · K_j: dS as 16-bit pairs in dP columns [0, 64)
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts_elect(tmem_base + kColDQ, tmem_base + kColDP + kk * 8,
                       dkmn + kslot + ((kk * 2048) >> 4), idesc_q, (jj > 0 || kk > 0) ? 1u : 0u);
        mma_commit_elect(bar_empty(kidx % S));
        mma_commit_elect(bar_acc_done);  // also orders the next S after this dQ MMA
      }
    }
    mma_commit_elect(bar_drain);
    mbar_wait_drain(bar_drain, 0, wc, kSiteDrain);
  } else {
    const int rho = warp * 32 + lane;
    const bool row_ok = rho < (i1 - i0) * p.group;
    const int qi = i0 + rho / p.group;
    const int h = g * p.group + rho % p.group;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const size_t vrow = (static_cast<size_t>(b) * p.Hq + h) * p.Lpad + min(qi, p.Lpad - 1);
    const float lse2 = row_ok ? p.lse2[vrow] : INFINITY;
    const float dsum = row_ok ? p.dsum[vrow] : 0.f;
    const int pos_min = i0, pos_max = i1 - 1;
    bool ok = true;
    for (int jj = 0; ok && jj < nblocks; ++jj) {
      const int key0 = (blk_lo + jj) * kBN;
      ok = mbar_wait_warp(bar_s_full, jj & 1u, wc, kSiteEw);
      if (!ok) break;
      tc_fence_after();
      const bool masked = (key0 + kBN > p.L) || (p.causal && key0 + kBN - 1 > pos_min) ||
                          (p.window_left >= 0 && key0 < pos_max - p.window_left) || !row_ok;
      int vis_lo = 0, vis_hi = kBN;
      if (masked) {
        const int hi_key = p.causal ? min(p.L, qi + 1) : p.L;
        const int lo_key = (p.window_left >= 0) ? qi - p.window_left : 0;
        vis_hi = row_ok ? max(0, min(kBN, hi_key - key0)) : 0;
        vis_lo = max(0, min(kBN, lo_key - key0));
      }
      elementwise_block<BF16, false>(tmem_base + lane_off + kColS, tmem_base + lane_off + kColDP,
                                     p.c2, vis_lo, vis_hi, masked,
                                     [&](int, float& l, float& d) { l = lse2; d = dsum; });
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p_full);
      // the next block's S overwrites these columns after the dQ MMA has read them
      if (jj + 1 < nblocks) {
        ok = mbar_wait_warp(bar_acc_done, jj & 1u, wc, kSiteEw);
      }
    }
    // epilogue: dQ · scale
    if (ok && nblocks > 0) {
      ok = mbar_wait_warp(bar_acc_done, (nblocks - 1) & 1u, wc, kSiteEw);
      if (ok) tc_fence_after();
    }
    if (ok && nblocks > 0) {
      const size_t off = ((static_cast<size_t>(b) * p.L + qi) * p.Hq + h) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t r[32];
        tmem_ld_x32(tmem_base + lane_off + kColDQ + c0, r);
        if (!row_ok) continue;
        if constexpr (OUT_F32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.dq) + off + c0);
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            dst[c >> 2] = make_float4(__uint_as_float(r[c]) * p.scale, __uint_as_float(r[c + 1]) * p.scale,
                                      __uint_as_float(r[c + 2]) * p.scale, __uint_as_float(r[c + 3]) * p.scale);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dq) + off + c0);
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint4 w;
            w.x = pack_in(__uint_as_float(r[c]) * p.scale, __uint_as_float(r[c + 1]) * p.scale, BF16);
            w.y = pack_in(__uint_as_float(r[c + 2]) * p.scale, __uint_as_float(r[c + 3]) * p.scale, BF16);
            w.z = pack_in(__uint_as_float(r[c + 4]) * p.scale, __uint_as_float(r[c + 5]) * p.scale, BF16);
            w.w = pack_in(__uint_as_float(r[c + 6]) * p.scale, __uint_as_float(r[c + 7]) * p.scale, BF16);
            dst[c >> 3] = w;
          }
        }
      }
    }
  }
  EX19_BWD_TEARDOWN()
}

// ----------------------------------------------------------------------- dK, dV
template <int D, bool BF16, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_lse2,
                         const __grid_constant__ CUtensorMap tm_dsum, const BwdParams p) {
  EX19_BWD_PREAMBLE()
  // item: (batch, K/V head, 128-key tile)
  const int nblk = (p.L + kBN - 1) / kBN;
  int x = blockIdx.x;
  const int jt = x % nblk;
  x /= nblk;
  const int g = x % p.Hkv, b = x / p.Hkv;
  const int k0 = jt * kBN;
  // query blocks whose rows see some key of this tile
  const int qb_lo = p.causal ? jt : 0;
  const int qb_hi = (p.window_left >= 0) ? min(nblk, (min(p.L, k0 + kBN) - 1 + p.window_left) / kBN + 1)
                                         : nblk;
  const int nq = max(0, qb_hi - qb_lo);
  const int nsteps = nq * p.group;  // (query head, query block) pairs
  // TMEM: Sᵀ [0,128), dPᵀ [128,256), dV [256, 256 + D), dK [256 + D, 256 + 2D)
  const uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;

  if (warp == kProducerWarp) {
    if (lane == 0 && nsteps > 0) {
      mbar_arrive_expect_tx(bar_res, 2 * G::kTileBytes);
      for (int c = 0; c < G::kChunks; ++c) {
        tma_load_4d(sRes + c * G::kChunkBytes, &tm_k, bar_res, c * 64, g, k0, b);
        tma_load_4d(sRes + G::kTileBytes + c * G::kChunkBytes, &tm_v, bar_res, c * 64, g, k0, b);
      }
      uint32_t n = 0;  // streamed tiles: Q then dO per step (pairs of slots)
      bool ok = true;
      for (int st = 0; ok && st < nsteps; ++st) {
        const int h = g * p.group + st / nq;
        const int ib = qb_lo + st % nq;
        for (int kv = 0; kv < 2; ++kv) {
          const uint32_t slot = n % S;
          ok = mbar_wait_bounded(bar_empty(slot), ((n / S) & 1u) ^ 1u, wc, kSiteProd);
          if (!ok) break;
          const uint32_t bytes = G::kTileBytes + (kv ? 0u : G::kVecBytes);
          mbar_arrive_expect_tx(bar_full(slot), bytes);
          for (int c = 0; c < G::kChunks; ++c)
            tma_load_4d(sRing + slot * G::kTileBytes + c * G::kChunkBytes, kv ? &tm_do : &tm_q,
                        bar_full(slot), c * 64, h, ib * kBM, b);
          if (kv == 0) {  // this step's LSE2 and D rows (128 floats each)
            const uint32_t vec = sVec + (slot / 2) * G::kVecBytes;
            tma_load_2d(vec, &tm_lse2, bar_full(slot), ib * kBM, b * p.Hq + h);
            tma_load_2d(vec + kBN * 4, &tm_dsum, bar_full(slot), ib * kBM, b * p.Hq + h);
          }
          ++n;
        }
      }
      if (!ok) {
        for (uint32_t back = 1; back <= S && back <= n; ++back) {
          const uint32_t m = n - back;
          mbar_wait_drain(bar_full(m % S), (m / S) & 1u, wc, kSiteDrain);
        }
        mbar_wait_drain(bar_res, 0, wc, kSiteDrain);
      }
    }
  } else if (warp == kMmaWarp) {
    if (nsteps > 0) {
      constexpr uint32_t idesc_s = idesc_f16_f32acc(BF16, kBM, kBN, false);
      constexpr uint32_t idesc_a = idesc_f16_f32acc(BF16, kBM, D, true);
      const uint64_t dk_ = sdesc_sw128(sRes, 16, 1024);                  // K_j, K-major
      const uint64_t dv_ = sdesc_sw128(sRes + G::kTileBytes, 16, 1024);  // V_j, K-major
      const uint64_t dr = sdesc_sw128(sRing, 16, 1024);                  // Q_i / dO_i, K-major
      const uint64_t drmn = sdesc_sw128(sRing, G::kChunkBytes, 1024);    // Q_i / dO_i, MN-major
      bool ok = mbar_wait_warp(bar_res, 0, wc, kSiteMma);
      for (int st = 0; ok && st < nsteps; ++st) {
        const uint32_t qidx = 2u * st, didx = qidx + 1u;
        ok = mbar_wait_warp(bar_full(qidx % S), (qidx / S) & 1u, wc, kSiteMma) &&
             mbar_wait_warp(bar_full(didx % S), (didx / S) & 1u, wc, kSiteMma);
        if (!ok) break;
        tc_fence_after();
        const uint64_t qs = ((qidx % S) * G::kTileBytes) >> 4;
        const uint64_t ds = ((didx % S) * G::kTileBytes) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * G::kChunkBytes + (kk & 3) * 32) >> 4;
          mma_ss_elect(tmem_base + kColS, dk_ + off, dr + qs + off, idesc_s, kk > 0);
          mma_ss_elect(tmem_base + kColDP, dv_ + off, dr + ds + off, idesc_s, kk > 0);
        }
        mma_commit_elect(bar_s_full);
        ok = mbar_wait_warp(bar_p_full, st & 1u, wc, kSiteMma);
        if (!ok) break;
        tc_fence_after();
        // dV += Pᵀ · dO_i and dK += dSᵀ · Q_i (16-bit pairs in columns [0,64) of Sᵀ / dPᵀ)
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk) {
          const uint32_t acc = (st > 0 || kk > 0) ? 1u : 0u;
          mma_ts_elect(tmem_base + kColDV, tmem_base + kColS + kk * 8,
                       drmn + ds + ((kk * 2048) >> 4), idesc_a, acc);
          mma_ts_elect(tmem_base + kColDK, tmem_base + kColDP + kk * 8,
                       drmn + qs + ((kk * 2048) >> 4), idesc_a, acc);
        }
        mma_commit_elect(bar_empty(qidx % S));
        mma_commit_elect(bar_empty(didx % S));
        mma_commit_elect(bar_acc_done);
      }
    }
    mma_commit_elect(bar_drain);
    mbar_wait_drain(bar_drain, 0, wc, kSiteDrain);
  } else {
    const int r = warp * 32 + lane;  // key row of the tile
    const int key = k0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    bool ok = true;
    for (int st = 0; ok && st < nsteps; ++st) {
      const int ib = qb_lo + st % nq;
      const int q0 = ib * kBM;
      ok = mbar_wait_warp(bar_s_full, st & 1u, wc, kSiteEw);
      if (!ok) break;
      tc_fence_after();
      // visible queries of this key row: q >= key (causal), q <= key + wl, q < L
      const bool masked = (key >= p.L) || (q0 + kBM > p.L) || (p.causal && q0 < k0 + kBN - 1) ||
                          (p.window_left >= 0 && q0 + kBM - 1 > k0 + p.window_left);
      int vis_lo = 0, vis_hi = kBM;
      if (masked) {
        int lo_q = p.causal ? key : 0;
        int hi_q = (p.window_left >= 0) ? key + p.window_left + 1 : p.L;
        hi_q = min(hi_q, p.L);
        if (key >= p.L) hi_q = lo_q = 0;
        vis_lo = max(0, min(kBM, lo_q - q0));
        vis_hi = max(0, min(kBM, hi_q - q0));
      }
      // this step's LSE2 and D rows: slot pair (2 st) / 2 of the ring's vector area
      const uint32_t vec = sVec + (((2u * st) % S) / 2) * G::kVecBytes;
      elementwise_block<BF16, true>(tmem_base + lane_off + kColS, tmem_base + lane_off + kColDP,
                                    p.c2, vis_lo, vis_hi, masked,
                                    [&](int c, float& l, float& d) {
                                      l = ld_shared_f32(vec + 4u * c);
                                      d = ld_shared_f32(vec + kBN * 4u + 4u * c);
                                    });
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p_full);
      ok = mbar_wait_warp(bar_acc_done, st & 1u, wc, kSiteEw);  // Sᵀ / dPᵀ reused next step
    }
    if (ok && nsteps > 0) {
      tc_fence_after();
      const bool row_ok = key < p.L;
      const size_t off = ((static_cast<size_t>(b) * p.L + key) * p.Hkv + g) * D;
#pragma unroll
      for (int which = 0; which < 2; ++which) {  // 0: dK (scaled), 1: dV
        void* out = which ? p.dv : p.dk;
        const float f = which ? 1.f : p.scale;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t rr[32];
          tmem_ld_x32(tmem_base + lane_off + (which ? kColDV : kColDK) + c0, rr);
          if (!row_ok) continue;
          if constexpr (OUT_F32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + off + c0);
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              dst[c >> 2] = make_float4(__uint_as_float(rr[c]) * f, __uint_as_float(rr[c + 1]) * f,
                                        __uint_as_float(rr[c + 2]) * f, __uint_as_float(rr[c + 3]) * f);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + off + c0);
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
              uint4 w;
              w.x = pack_in(__uint_as_float(rr[c]) * f, __uint_as_float(rr[c + 1]) * f, BF16);
              w.y = pack_in(__uint_as_float(rr[c + 2]) * f, __uint_as_float(rr[c + 3]) * f, BF16);
              w.z = pack_in(__uint_as_float(rr[c + 4]) * f, __uint_as_float(rr[c + 5]) * f, BF16);
              w.w = pack_in(__uint_as_float(rr[c + 6]) * f, __uint_as_float(rr[c + 7]) * f, BF16);
              dst[c >> 3] = w;
            }
          }
        }
      }
    }
    if (ok && nsteps == 0 && key < p.L) {
      // no query sees these keys: zero gradients
      const size_t off = ((static_cast<size_t>(b) * p.L + key) * p.Hkv + g) * D;
      for (int c = 0; c < D; ++c) {
        if constexpr (OUT_F32) {
          static_cast<float*>(p.dk)[off + c] = 0.f;
          static_cast<float*>(p.dv)[off + c] = 0.f;
        } else {
          static_cast<uint16_t*>(p.dk)[off + c] = 0;
          static_cast<uint16_t*>(p.dv)[off + c] = 0;
        }
      }
    }
  }
  EX19_BWD_TEARDOWN()
}

#undef EX19_BWD_PREAMBLE
#undef EX19_BWD_TEARDOWN

}  // namespace bwd
}  // namespace ex19
