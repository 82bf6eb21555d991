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
// GB300 mapping: three kernels, each with 8 elementwise warps in two groups of 4
// (group h owns columns [64h, 64h + 64) of every 128 x 128 block, the warp's lane
// quarter owns 32 rows), one TMA producer warp and two MMA warps, one issuing the
// S / dP products and one the accumulating products, so that neither stream of
// MMAs waits behind the other's barrier; every wait bounded:
//   * attn_bwd_prep: D and LSE2 per row into the workspace.
//   * attn_bwd_dq_kernel (query-stationary, one CTA per 128-row tile packed as in
//     the one-tile forward): per key block, S = Q Kᵀ and dP = dO Vᵀ (SS MMAs into
//     TMEM, issued per 64-key half), dS written as 16-bit pairs into one of two dS
//     buffers, then dQ += dS · K (A = dS from TMEM, B = K MN-major in shared memory).
//   * attn_bwd_dkdv_kernel (key-stationary, one CTA per (batch, K/V head, 128-key
//     tile)): per (query head of the group, query block), Sᵀ = K Qᵀ and dPᵀ = V dOᵀ,
//     Pᵀ and dSᵀ written as 16-bit pairs, then dV += Pᵀ · dO and dK += dSᵀ · Q.
// Overlap: a group releases its half of the S / dP columns as soon as it has loaded
// them into registers, and the MMA warp issues the next block's S and dP half into
// them at once, so the tensor core computes block j + 1 while the elementwise warps
// work on block j. The accumulating MMAs are split the same way (K = the group's 64
// keys or queries), so the issue order per block is: half 0 of block j + 1, group 0's
// share of block j, half 1 of block j + 1, group 1's share of block j; each waits
// only for its own group. The 16-bit results go to separate TMEM buffers (dQ kernel:
// two per group, dK/dV kernel at d = 64: one); at d = 128 the dK/dV kernel has no
// TMEM left for them (Sᵀ, dPᵀ, dV, dK fill 512 columns), writes Pᵀ and dSᵀ over the
// columns it has read, and issues a half of the next step after that group's share.
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
constexpr int kEwWarps = 8;
constexpr int kThreads = 32 * (kEwWarps + 3);  // elementwise warps + producer + two MMA warps
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;   // S / dP MMAs (and the TMEM allocation)
constexpr int kAccWarp = 10;  // accumulating MMAs (dQ, or dV and dK)
constexpr int kHalfN = 64;      // columns per elementwise group (and per S / dP MMA half)
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
  static constexpr int kHalfRows = kHalfN * 128;    // byte offset of row 64 in a chunk
  static constexpr int kSlots = (D == 64) ? 8 : 4;  // streamed tiles
  static constexpr int kOffRes = 0;                 // 2 resident tiles
  static constexpr int kOffRing = 2 * kTileBytes;
  static constexpr int kOffVec = kOffRing + kSlots * kTileBytes;  // dK/dV kernel: LSE2, D rows
  static constexpr int kVecBytes = 2 * kBN * 4;                   // per stage
  static constexpr int kOffBar = kOffVec + (kSlots / 2) * kVecBytes;
  // barriers: full[S], empty[S], res_full, s_full[2], ld_free[2], p_full[2][2],
  // acc_done[2][2], drain, a_ready
  static constexpr int kNumBars = 2 * kSlots + 15;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemUsed = kOffMisc + 16;
  static constexpr int kSmemBytes = kSmemUsed + 1024;
};

// The 16-bit pair of a fp32 pair in the input dtype.
__device__ __forceinline__ uint32_t pack_in(float a, float b, bool bf16) { return pack2(a, b, bf16); }

__device__ __forceinline__ float4 ld_shared_v4f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// Two tcgen05.ld (32x32b) of N columns each and one tcgen05.wait::ld, in one asm
// statement so that no use of the registers is scheduled before the data arrives.
__device__ __forceinline__ void tmem_ld2_x32(uint32_t ta, uint32_t (&ra)[32], uint32_t tb,
                                               uint32_t (&rb)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(ra[0]), "=r"(ra[1]), "=r"(ra[2]), "=r"(ra[3]), "=r"(ra[4]), "=r"(ra[5]), "=r"(ra[6]), "=r"(ra[7]), "=r"(ra[8]), "=r"(ra[9]), "=r"(ra[10]), "=r"(ra[11]), "=r"(ra[12]), "=r"(ra[13]), "=r"(ra[14]), "=r"(ra[15]), "=r"(ra[16]), "=r"(ra[17]), "=r"(ra[18]), "=r"(ra[19]), "=r"(ra[20]), "=r"(ra[21]), "=r"(ra[22]), "=r"(ra[23]), "=r"(ra[24]), "=r"(ra[25]), "=r"(ra[26]), "=r"(ra[27]), "=r"(ra[28]), "=r"(ra[29]), "=r"(ra[30]), "=r"(ra[31]), "=r"(rb[0]), "=r"(rb[1]), "=r"(rb[2]), "=r"(rb[3]), "=r"(rb[4]), "=r"(rb[5]), "=r"(rb[6]), "=r"(rb[7]), "=r"(rb[8]), "=r"(rb[9]), "=r"(rb[10]), "=r"(rb[11]), "=r"(rb[12]), "=r"(rb[13]), "=r"(rb[14]), "=r"(rb[15]), "=r"(rb[16]), "=r"(rb[17]), "=r"(rb[18]), "=r"(rb[19]), "=r"(rb[20]), "=r"(rb[21]), "=r"(rb[22]), "=r"(rb[23]), "=r"(rb[24]), "=r"(rb[25]), "=r"(rb[26]), "=r"(rb[27]), "=r"(rb[28]), "=r"(rb[29]), "=r"(rb[30]), "=r"(rb[31])
      : "r"(ta), "r"(tb)
      : "memory");
}

__device__ __forceinline__ void tmem_ld2_x64(uint32_t ta, uint32_t (&ra)[64], uint32_t tb,
                                               uint32_t (&rb)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%128];\n"
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%129];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(ra[0]), "=r"(ra[1]), "=r"(ra[2]), "=r"(ra[3]), "=r"(ra[4]), "=r"(ra[5]), "=r"(ra[6]), "=r"(ra[7]), "=r"(ra[8]), "=r"(ra[9]), "=r"(ra[10]), "=r"(ra[11]), "=r"(ra[12]), "=r"(ra[13]), "=r"(ra[14]), "=r"(ra[15]), "=r"(ra[16]), "=r"(ra[17]), "=r"(ra[18]), "=r"(ra[19]), "=r"(ra[20]), "=r"(ra[21]), "=r"(ra[22]), "=r"(ra[23]), "=r"(ra[24]), "=r"(ra[25]), "=r"(ra[26]), "=r"(ra[27]), "=r"(ra[28]), "=r"(ra[29]), "=r"(ra[30]), "=r"(ra[31]), "=r"(ra[32]), "=r"(ra[33]), "=r"(ra[34]), "=r"(ra[35]), "=r"(ra[36]), "=r"(ra[37]), "=r"(ra[38]), "=r"(ra[39]), "=r"(ra[40]), "=r"(ra[41]), "=r"(ra[42]), "=r"(ra[43]), "=r"(ra[44]), "=r"(ra[45]), "=r"(ra[46]), "=r"(ra[47]), "=r"(ra[48]), "=r"(ra[49]), "=r"(ra[50]), "=r"(ra[51]), "=r"(ra[52]), "=r"(ra[53]), "=r"(ra[54]), "=r"(ra[55]), "=r"(ra[56]), "=r"(ra[57]), "=r"(ra[58]), "=r"(ra[59]), "=r"(ra[60]), "=r"(ra[61]), "=r"(ra[62]), "=r"(ra[63]), "=r"(rb[0]), "=r"(rb[1]), "=r"(rb[2]), "=r"(rb[3]), "=r"(rb[4]), "=r"(rb[5]), "=r"(rb[6]), "=r"(rb[7]), "=r"(rb[8]), "=r"(rb[9]), "=r"(rb[10]), "=r"(rb[11]), "=r"(rb[12]), "=r"(rb[13]), "=r"(rb[14]), "=r"(rb[15]), "=r"(rb[16]), "=r"(rb[17]), "=r"(rb[18]), "=r"(rb[19]), "=r"(rb[20]), "=r"(rb[21]), "=r"(rb[22]), "=r"(rb[23]), "=r"(rb[24]), "=r"(rb[25]), "=r"(rb[26]), "=r"(rb[27]), "=r"(rb[28]), "=r"(rb[29]), "=r"(rb[30]), "=r"(rb[31]), "=r"(rb[32]), "=r"(rb[33]), "=r"(rb[34]), "=r"(rb[35]), "=r"(rb[36]), "=r"(rb[37]), "=r"(rb[38]), "=r"(rb[39]), "=r"(rb[40]), "=r"(rb[41]), "=r"(rb[42]), "=r"(rb[43]), "=r"(rb[44]), "=r"(rb[45]), "=r"(rb[46]), "=r"(rb[47]), "=r"(rb[48]), "=r"(rb[49]), "=r"(rb[50]), "=r"(rb[51]), "=r"(rb[52]), "=r"(rb[53]), "=r"(rb[54]), "=r"(rb[55]), "=r"(rb[56]), "=r"(rb[57]), "=r"(rb[58]), "=r"(rb[59]), "=r"(rb[60]), "=r"(rb[61]), "=r"(rb[62]), "=r"(rb[63])
      : "r"(ta), "r"(tb)
      : "memory");
}

// Common preamble of both kernels: barriers, TMEM, wait control.
//   s_full[h]   MMA -> group h: the block's S and dP columns of half h are written
//   ld_free[h]  group h -> MMA: half h of S and dP is in registers (128 arrivals)
//   p_full[h][b]   group h -> MMA: its 16-bit results in buffer b are written (128 arrivals)
//   acc_done[h][b] MMA -> group h: the accumulating MMAs that read them are complete
//   drain          MMA -> all: every MMA of the CTA is complete (both MMA warps commit;
//                  the epilogues wait here)
//   a_ready        elementwise -> MMA: resident tiles copied into TMEM (d = 64)
// A slot read by both MMA warps is released by two commits: EMPTY_EVEN / EMPTY_ODD
// arrivals for the even (K or Q) and odd (V or dO) slots.
#define EX19_BWD_PREAMBLE(EMPTY_EVEN, EMPTY_ODD)                                               \
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
  auto bar_s_full = [&](uint32_t h) { return bars + 8u * (2 * S + 1 + h); };                   \
  auto bar_ld_free = [&](uint32_t h) { return bars + 8u * (2 * S + 3 + h); };                  \
  auto bar_p_full = [&](uint32_t h, uint32_t b) { return bars + 8u * (2 * S + 5 + 2 * h + b); }; \
  auto bar_acc_done = [&](uint32_t h, uint32_t b) { return bars + 8u * (2 * S + 9 + 2 * h + b); }; \
  const uint32_t bar_drain = bars + 8u * (2 * S + 13);                                         \
  const uint32_t bar_a_ready = bars + 8u * (2 * S + 14);                                       \
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::kOffMisc);                       \
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + G::kOffMisc + 4); \
  const int warp = threadIdx.x >> 5;                                                           \
  const int lane = threadIdx.x & 31;                                                           \
  if (threadIdx.x == 0) {                                                                      \
    for (int s = 0; s < S; ++s) {                                                              \
      mbar_init(bar_full(s), 1);                                                               \
      mbar_init(bar_empty(s), (s & 1) ? (EMPTY_ODD) : (EMPTY_EVEN));                           \
    }                                                                                          \
    mbar_init(bar_res, 1);                                                                     \
    for (int k = 0; k < 2; ++k) {                                                              \
      mbar_init(bar_s_full(k), 1);                                                             \
      mbar_init(bar_ld_free(k), 4 * 32);                                                       \
      for (int b2 = 0; b2 < 2; ++b2) {                                                         \
        mbar_init(bar_p_full(k, b2), 4 * 32);                                                  \
        mbar_init(bar_acc_done(k, b2), 1);                                                     \
      }                                                                                        \
    }                                                                                          \
    mbar_init(bar_drain, 2);                                                                   \
    mbar_init(bar_a_ready, kEwWarps * 32);                                                     \
    *abort_flag = 0u;                                                                          \
    fence_mbar_init();                                                                         \
  }                                                                                            \
  /* launched as a programmatic dependent: the kernels before it on the stream have */         \
  /* completed and their writes are visible past this point (no-op otherwise); TMEM */        \
  /* is allocated only after it, so no CTA holds TMEM while it waits on another kernel */      \
  asm volatile("griddepcontrol.wait;" ::: "memory");                                           \
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
  wc.set_limit(p.wait_limit_ns);                                                               \
  wc.unit = blockIdx.x;

#define EX19_BWD_TEARDOWN()            \
  tc_fence_before();                   \
  __syncthreads();                     \
  tc_fence_after();                    \
  if (warp == kMmaWarp) {              \
    __syncwarp();                      \
    tmem_dealloc(tmem_base, kTmemCols); \
  }

// Elementwise pass of N columns x0 .. x0+N-1 of a block, from the thread's row of X
// (S or Sᵀ, fp32) and dX (dP or dPᵀ) already in registers:
// W = 2^(X·c − lse2[col]) (0 outside [vis_lo, vis_hi)), dS = W (dX − dsum[col]),
// both as 16-bit pairs (W only if kW). lse2 / dsum of four columns at a time come
// from `vec4(col, l, d)` (dK/dV kernel: shared memory) or are the row's own values.
template <int N, bool BF16, bool kW, bool kMasked, typename Vec4Fn>
__device__ __forceinline__ void elementwise_cols(const uint32_t (&xs)[N], const uint32_t (&dxs)[N],
                                                 int x0, float c2, int vis_lo, int vis_hi, Vec4Fn vec4,
                                                 uint32_t* wpk, uint32_t* dspk) {
  // paired fp32 arithmetic (one FFMA2 / FADD2 / FMUL2 per two columns; each lane
  // rounds as the scalar operation would)
  const float2 c22 = make_float2(c2, c2);
#pragma unroll
  for (int c = 0; c < N; c += 4) {
    float l[4], d[4];
    vec4(x0 + c, l, d);
#pragma unroll
    for (int u = 0; u < 4; u += 2) {
      const float2 a = __ffma2_rn(make_float2(__uint_as_float(xs[c + u]), __uint_as_float(xs[c + u + 1])),
                                  c22, make_float2(-l[u], -l[u + 1]));
      float w0 = ex2_approx(a.x), w1 = ex2_approx(a.y);
      if constexpr (kMasked) {
        const int cc = x0 + c + u;
        w0 = (cc >= vis_lo && cc < vis_hi) ? w0 : 0.f;
        w1 = (cc + 1 >= vis_lo && cc + 1 < vis_hi) ? w1 : 0.f;
      }
      const float2 dd = __fadd2_rn(make_float2(__uint_as_float(dxs[c + u]), __uint_as_float(dxs[c + u + 1])),
                                   make_float2(-d[u], -d[u + 1]));
      const float2 sv = __fmul2_rn(make_float2(w0, w1), dd);
      if constexpr (kW) wpk[(c + u) >> 1] = pack_in(w0, w1, BF16);
      dspk[(c + u) >> 1] = pack_in(sv.x, sv.y, BF16);
    }
  }
}

// Copies row r of a 128 x 64 16-bit tile in the 128-byte swizzle (16-byte chunk c of
// row r at chunk c ^ (r mod 8)) into the thread's TMEM lane as 32 columns of pairs:
// the layout of a TMEM A operand (K-step kk at columns 8 kk .. 8 kk + 7).
__device__ __forceinline__ void tile_row_to_tmem64(uint32_t s_tile, int r, uint32_t taddr) {
  uint32_t v[32];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t a = s_tile + r * 128 + ((c ^ (r & 7)) << 4);
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[4 * c]), "=r"(v[4 * c + 1]), "=r"(v[4 * c + 2]), "=r"(v[4 * c + 3])
                 : "r"(a));
  }
  tmem_st_x32(taddr, v);
}

// Writes columns [c_lo, c_lo + D/2) of the thread's row of a TMEM fp32 accumulator,
// times f, to out (input dtype or float32).
template <int D, bool BF16, bool OUT_F32>
__device__ __forceinline__ void store_acc_half(uint32_t tacc, int c_lo, float f, bool row_ok, void* out,
                                               size_t off) {
#pragma unroll
  for (int c0 = 0; c0 < D / 2; c0 += 32) {
    uint32_t r[32];
    tmem_ld_x32(tacc + c_lo + c0, r);
    if (!row_ok) continue;
    if constexpr (OUT_F32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + off + c_lo + c0);
#pragma unroll
      for (int c = 0; c < 32; c += 4)
        dst[c >> 2] = make_float4(__uint_as_float(r[c]) * f, __uint_as_float(r[c + 1]) * f,
                                  __uint_as_float(r[c + 2]) * f, __uint_as_float(r[c + 3]) * f);
    } else {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + off + c_lo + c0);
#pragma unroll
      for (int c = 0; c < 32; c += 8) {
        uint4 w;
        w.x = pack_in(__uint_as_float(r[c]) * f, __uint_as_float(r[c + 1]) * f, BF16);
        w.y = pack_in(__uint_as_float(r[c + 2]) * f, __uint_as_float(r[c + 3]) * f, BF16);
        w.z = pack_in(__uint_as_float(r[c + 4]) * f, __uint_as_float(r[c + 5]) * f, BF16);
        w.w = pack_in(__uint_as_float(r[c + 6]) * f, __uint_as_float(r[c + 7]) * f, BF16);
        dst[c >> 3] = w;
      }
    }
  }
}

// ------------------------------------------------------------------------- dQ
template <int D, bool BF16, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const BwdParams p) {
  EX19_BWD_PREAMBLE(2, 1)  // K_j: S (MMA warp) and dQ (accumulating warp); V_j: dP only
  // item: (batch, K/V head, packed row tile), the last row tiles (most key blocks
  // when causal) first so that the short ones fill the end of the grid
  const int nbg = p.B * p.Hkv;
  const int rt = p.row_tiles - 1 - static_cast<int>(blockIdx.x) / nbg;
  const int g = static_cast<int>(blockIdx.x) % nbg % p.Hkv, b = static_cast<int>(blockIdx.x) % nbg / p.Hkv;
  const int i0 = rt * p.q_per_tile, i1 = min(p.L, i0 + p.q_per_tile);
  const int nblk = (p.L + kBN - 1) / kBN;
  const int blk_hi = p.causal ? (i1 - 1) / kBN + 1 : nblk;
  const int blk_lo = (p.window_left >= 0) ? max(0, i0 - p.window_left) / kBN : 0;
  const int nblocks = max(0, blk_hi - blk_lo);
  // TMEM: S [0,128), dP [128,256), dQ [256, 256 + D), dS buffers of 64 columns after dQ;
  // d = 64: Q [448, 480) and dO [480, 512) as A operands, so that S and dP are TS
  // MMAs reading only K and V from shared memory
  constexpr bool kATmem = (D == 64);
  const uint32_t kColS = 0, kColDP = 128, kColDQ = 256;
  constexpr uint32_t kColQ = 448, kColDO = 480;
  auto col_ds = [](uint32_t buf) { return 256u + D + 64u * buf; };

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
      // Whether or not this CTA aborted, the copies issued last may still be in
      // flight (another role can abort after this loop has ended, and then nothing
      // consumes them): let them land before the CTA can exit.
      {
        for (uint32_t back = 1; back <= S && back <= n; ++back) {
          const uint32_t m = n - back;
          mbar_wait_drain(bar_full(m % S), (m / S) & 1u, wc, kSiteDrain);
        }
        mbar_wait_drain(bar_res, 0, wc, kSiteDrain);
      }
    }
  } else if (warp == kMmaWarp) {
    if (nblocks > 0) {
      constexpr uint32_t idesc_s = idesc_f16_f32acc(BF16, kBM, kHalfN, false);
      const uint64_t dq_ = sdesc_sw128(sRes, 16, 1024);                   // Q, K-major
      const uint64_t ddo = sdesc_sw128(sRes + G::kTileBytes, 16, 1024);   // dO, K-major
      const uint64_t dkv = sdesc_sw128(sRing, 16, 1024);                  // K / V, K-major
      // S and dP of block jj, keys [64h, 64h + 64): N = 64 MMAs into columns 64h..
      auto issue_half = [&](int jj, int hh) __attribute__((always_inline)) -> bool {
        const uint32_t kidx = 2u * jj, vidx = kidx + 1u;
        if (hh == 0) {
          if (!mbar_wait_warp(bar_full(kidx % S), (kidx / S) & 1u, wc, kSiteMma) ||
              !mbar_wait_warp(bar_full(vidx % S), (vidx / S) & 1u, wc, kSiteMma))
            return false;
        }
        tc_fence_after();
        const uint64_t kslot = ((kidx % S) * G::kTileBytes + hh * G::kHalfRows) >> 4;
        const uint64_t vslot = ((vidx % S) * G::kTileBytes + hh * G::kHalfRows) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * G::kChunkBytes + (kk & 3) * 32) >> 4;
          if constexpr (kATmem) {
            mma_ts_elect(tmem_base + kColS + kHalfN * hh, tmem_base + kColQ + kk * 8, dkv + kslot + off,
                         idesc_s, kk > 0);
            mma_ts_elect(tmem_base + kColDP + kHalfN * hh, tmem_base + kColDO + kk * 8, dkv + vslot + off,
                         idesc_s, kk > 0);
          } else {
            mma_ss_elect(tmem_base + kColS + kHalfN * hh, dq_ + off, dkv + kslot + off, idesc_s, kk > 0);
            mma_ss_elect(tmem_base + kColDP + kHalfN * hh, ddo + off, dkv + vslot + off, idesc_s, kk > 0);
          }
        }
        mma_commit_elect(bar_s_full(hh));
        if (hh == 1) {
          mma_commit_elect(bar_empty(vidx % S));  // V_j is only read by dP
          mma_commit_elect(bar_empty(kidx % S));  // this warp's share of K_j
        }
        return true;
      };
      bool ok = kATmem ? mbar_wait_warp(bar_a_ready, 0, wc, kSiteMma) : mbar_wait_warp(bar_res, 0, wc, kSiteMma);
      if (ok) {
        tc_fence_after();
        ok = issue_half(0, 0) && issue_half(0, 1);
      }
      // half hh of block jj + 1 as soon as group hh has read its half of block jj
      for (int jj = 0; ok && jj + 1 < nblocks; ++jj)
        for (int hh = 0; ok && hh < 2; ++hh)
          ok = mbar_wait_warp(bar_ld_free(hh), jj & 1u, wc, kSiteMma) && issue_half(jj + 1, hh);
    }
    mma_commit_elect(bar_drain);
    mbar_wait_drain(bar_drain, 0, wc, kSiteDrain);
  } else if (warp == kAccWarp) {
    if (nblocks > 0) {
      constexpr uint32_t idesc_q = idesc_f16_f32acc(BF16, kBM, D, true);
      const uint64_t dkmn = sdesc_sw128(sRing, G::kChunkBytes, 1024);     // K, MN-major
      bool ok = true;
      for (int jj = 0; ok && jj < nblocks; ++jj) {
        const uint32_t buf = jj & 1;
        const uint32_t kidx = 2u * jj;
        const uint64_t kslot = ((kidx % S) * G::kTileBytes) >> 4;
        for (int hh = 0; ok && hh < 2; ++hh) {
          // dQ += dS[:, keys of half hh] · K_j[keys of half hh]: group hh's dS pairs sit in
          // columns 32 hh .. 32 hh + 31 of dS buffer `buf`
          ok = mbar_wait_warp(bar_p_full(hh, buf), (jj >> 1) & 1u, wc, kSiteMma);
          // K_j's load (complete long before: S_j was computed from it); this warp holds
          // the slot until its commit below, so the phase cannot move on
          if (ok && hh == 0) ok = mbar_wait_warp(bar_full(kidx % S), (kidx / S) & 1u, wc, kSiteMma);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k4 = 0; k4 < kHalfN / 16; ++k4) {
            const int kk = 4 * hh + k4;
            mma_ts_elect(tmem_base + kColDQ, tmem_base + col_ds(buf) + kk * 8,
                         dkmn + kslot + ((kk * 2048) >> 4), idesc_q, (jj > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_elect(bar_acc_done(hh, buf));
        }
        if (!ok) break;
        mma_commit_elect(bar_empty(kidx % S));
      }
    }
    mma_commit_elect(bar_drain);
    mbar_wait_drain(bar_drain, 0, wc, kSiteDrain);
  } else {
    const int hh = warp >> 2;                   // column half of this warp's group
    const int rho = (warp & 3) * 32 + lane;     // row of the tile
    const bool row_ok = rho < (i1 - i0) * p.group;
    const int qi = i0 + rho / p.group;
    const int h = g * p.group + rho % p.group;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const size_t vrow = (static_cast<size_t>(b) * p.Hq + h) * p.Lpad + min(qi, p.Lpad - 1);
    const float lse2 = row_ok ? p.lse2[vrow] : INFINITY;
    const float dsum = row_ok ? p.dsum[vrow] : 0.f;
    const int pos_min = i0, pos_max = i1 - 1;
    const int x0 = kHalfN * hh;
    bool ok = true;
    if constexpr (kATmem) {  // group 0 copies Q, group 1 dO, into their TMEM columns
      if (nblocks > 0) {
        ok = mbar_wait_warp(bar_res, 0, wc, kSiteEw);
        if (ok) {
          tile_row_to_tmem64(sRes + hh * G::kTileBytes, rho, tmem_base + lane_off + (hh ? kColDO : kColQ));
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar_a_ready);
        }
      }
    }
    for (int jj = 0; ok && jj < nblocks; ++jj) {
      const int key0 = (blk_lo + jj) * kBN;
      const uint32_t buf = jj & 1;
      ok = mbar_wait_warp(bar_s_full(hh), jj & 1u, wc, kSiteEw);
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
      uint32_t dspk[32];
      {
        uint32_t xs[64], dxs[64];
        tmem_ld2_x64(tmem_base + lane_off + kColS + x0, xs, tmem_base + lane_off + kColDP + x0, dxs);
        tc_fence_before();
        mbar_arrive(bar_ld_free(hh));  // these columns may take the next block
        auto vec4 = [&](int, float (&l)[4], float (&d)[4]) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            l[u] = lse2;
            d[u] = dsum;
          }
        };
        // warp-uniform choice (the masked path is exact for every lane)
        if (__any_sync(0xffffffffu, masked))
          elementwise_cols<64, BF16, false, true>(xs, dxs, x0, p.c2, vis_lo, vis_hi, vec4, nullptr, dspk);
        else
          elementwise_cols<64, BF16, false, false>(xs, dxs, x0, p.c2, vis_lo, vis_hi, vec4, nullptr, dspk);
      }
      // this group's part of dS buffer `buf` was read by its dQ MMAs of block jj - 2
      if (jj >= 2) {
        ok = mbar_wait_warp(bar_acc_done(hh, buf), ((jj - 2) >> 1) & 1u, wc, kSiteEw);
        if (!ok) break;
        tc_fence_after();
      }
      tmem_st_x32(tmem_base + lane_off + col_ds(buf) + 32 * hh, dspk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p_full(hh, buf));
    }
    // epilogue: dQ · scale once every MMA is complete (both groups' shares);
    // group h writes columns [h D/2, (h + 1) D/2)
    if (ok && nblocks > 0) {
      ok = mbar_wait_warp(bar_drain, 0, wc, kSiteEw);
      if (ok) tc_fence_after();
    }
    if (ok && nblocks > 0) {
      const size_t off = ((static_cast<size_t>(b) * p.L + qi) * p.Hq + h) * D;
      store_acc_half<D, BF16, OUT_F32>(tmem_base + lane_off + kColDQ, hh * (D / 2), p.scale, row_ok,
                                       p.dq, off);
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
  EX19_BWD_PREAMBLE(2, 2)  // Q_i and dO_i are read by both MMA warps
  // Pᵀ and dSᵀ in their own TMEM columns (block st + 1 overlaps block st), or over
  // the columns of Sᵀ and dPᵀ that hold them (no room at d = 128)
  constexpr bool kSeparate = (D == 64);
  // item: (batch, K/V head, 128-key tile), the first key tiles (most query blocks
  // when causal) first so that the short ones fill the end of the grid
  const int nblk = (p.L + kBN - 1) / kBN;
  const int nbg = p.B * p.Hkv;
  const int jt = static_cast<int>(blockIdx.x) / nbg;
  const int g = static_cast<int>(blockIdx.x) % nbg % p.Hkv, b = static_cast<int>(blockIdx.x) % nbg / p.Hkv;
  const int k0 = jt * kBN;
  // query blocks whose rows see some key of this tile
  const int qb_lo = p.causal ? jt : 0;
  const int qb_hi = (p.window_left >= 0) ? min(nblk, (min(p.L, k0 + kBN) - 1 + p.window_left) / kBN + 1)
                                         : nblk;
  const int nq = max(0, qb_hi - qb_lo);
  const int nsteps = nq * p.group;  // (query head, query block) pairs
  // TMEM: Sᵀ [0,128), dPᵀ [128,256), dV [256, 256 + D), dK [256 + D, 256 + 2D);
  // d = 64: Pᵀ [384, 448), dSᵀ [448, 512). In place: group h's 16-bit results for
  // queries [64h, 64h + 64) at columns 64h .. 64h + 31 of Sᵀ and of dPᵀ.
  const uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  constexpr uint32_t kColPT = kSeparate ? 384u : 0u, kColDST = kSeparate ? 448u : 128u;
  // TMEM column of the 16-bit operand pairs for queries [16 kk, 16 kk + 16)
  auto op_col = [](uint32_t base, int kk) -> uint32_t {
    return kSeparate ? base + kk * 8 : base + (kk >> 2) * kHalfN + (kk & 3) * 8;
  };

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
      // Whether or not this CTA aborted, the copies issued last may still be in
      // flight (another role can abort after this loop has ended, and then nothing
      // consumes them): let them land before the CTA can exit.
      {
        for (uint32_t back = 1; back <= S && back <= n; ++back) {
          const uint32_t m = n - back;
          mbar_wait_drain(bar_full(m % S), (m / S) & 1u, wc, kSiteDrain);
        }
        mbar_wait_drain(bar_res, 0, wc, kSiteDrain);
      }
    }
  } else if (warp == kMmaWarp) {
    if (nsteps > 0) {
      constexpr uint32_t idesc_s = idesc_f16_f32acc(BF16, kBM, kHalfN, false);
      const uint64_t dk_ = sdesc_sw128(sRes, 16, 1024);                  // K_j, K-major
      const uint64_t dv_ = sdesc_sw128(sRes + G::kTileBytes, 16, 1024);  // V_j, K-major
      const uint64_t dr = sdesc_sw128(sRing, 16, 1024);                  // Q_i / dO_i, K-major
      // Sᵀ and dPᵀ of step st, queries [64h, 64h + 64): N = 64 MMAs into columns 64h..
      auto issue_half = [&](int st, int hh) __attribute__((always_inline)) -> bool {
        const uint32_t qidx = 2u * st, didx = qidx + 1u;
        if (hh == 0) {
          if (!mbar_wait_warp(bar_full(qidx % S), (qidx / S) & 1u, wc, kSiteMma) ||
              !mbar_wait_warp(bar_full(didx % S), (didx / S) & 1u, wc, kSiteMma))
            return false;
        }
        tc_fence_after();
        const uint64_t qs = ((qidx % S) * G::kTileBytes + hh * G::kHalfRows) >> 4;
        const uint64_t ds = ((didx % S) * G::kTileBytes + hh * G::kHalfRows) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * G::kChunkBytes + (kk & 3) * 32) >> 4;
          mma_ss_elect(tmem_base + kColS + kHalfN * hh, dk_ + off, dr + qs + off, idesc_s, kk > 0);
          mma_ss_elect(tmem_base + kColDP + kHalfN * hh, dv_ + off, dr + ds + off, idesc_s, kk > 0);
        }
        mma_commit_elect(bar_s_full(hh));
        if (hh == 1) {  // this warp's share of Q_i and dO_i
          mma_commit_elect(bar_empty(qidx % S));
          mma_commit_elect(bar_empty(didx % S));
        }
        return true;
      };
      bool ok = mbar_wait_warp(bar_res, 0, wc, kSiteMma);
      if (ok) {
        tc_fence_after();
        ok = issue_half(0, 0) && issue_half(0, 1);
      }
      // half hh of step st + 1 once group hh has read step st (separate buffers), or
      // once the accumulating MMAs that read group hh's pairs in place are complete
      for (int st = 0; ok && st + 1 < nsteps; ++st)
        for (int hh = 0; ok && hh < 2; ++hh) {
          ok = kSeparate ? mbar_wait_warp(bar_ld_free(hh), st & 1u, wc, kSiteMma)
                         : mbar_wait_warp(bar_acc_done(hh, 0), st & 1u, wc, kSiteMma);
          ok = ok && issue_half(st + 1, hh);
        }
    }
    mma_commit_elect(bar_drain);
    mbar_wait_drain(bar_drain, 0, wc, kSiteDrain);
  } else if (warp == kAccWarp) {
    if (nsteps > 0) {
      constexpr uint32_t idesc_a = idesc_f16_f32acc(BF16, kBM, D, true);
      const uint64_t drmn = sdesc_sw128(sRing, G::kChunkBytes, 1024);    // Q_i / dO_i, MN-major
      bool ok = true;
      for (int st = 0; ok && st < nsteps; ++st) {
        const uint32_t qidx = 2u * st, didx = qidx + 1u;
        const uint64_t qs = ((qidx % S) * G::kTileBytes) >> 4;
        const uint64_t ds = ((didx % S) * G::kTileBytes) >> 4;
        for (int hh = 0; ok && hh < 2; ++hh) {
          ok = mbar_wait_warp(bar_p_full(hh, 0), st & 1u, wc, kSiteMma);
          // Q_i and dO_i loads (complete long before: Sᵀ and dPᵀ were computed from
          // them); this warp holds both slots until its commits below
          if (ok && hh == 0)
            ok = mbar_wait_warp(bar_full(qidx % S), (qidx / S) & 1u, wc, kSiteMma) &&
                 mbar_wait_warp(bar_full(didx % S), (didx / S) & 1u, wc, kSiteMma);
          if (!ok) break;
          tc_fence_after();
          // dV += Pᵀ · dO_i and dK += dSᵀ · Q_i over the queries of half hh (group hh's pairs)
#pragma unroll
          for (int k4 = 0; k4 < kHalfN / 16; ++k4) {
            const int kk = 4 * hh + k4;
            const uint32_t acc = (st > 0 || kk > 0) ? 1u : 0u;
            mma_ts_elect(tmem_base + kColDV, tmem_base + op_col(kColPT, kk),
                         drmn + ds + ((kk * 2048) >> 4), idesc_a, acc);
            mma_ts_elect(tmem_base + kColDK, tmem_base + op_col(kColDST, kk),
                         drmn + qs + ((kk * 2048) >> 4), idesc_a, acc);
          }
          mma_commit_elect(bar_acc_done(hh, 0));
        }
        if (!ok) break;
        mma_commit_elect(bar_empty(qidx % S));
        mma_commit_elect(bar_empty(didx % S));
      }
    }
    mma_commit_elect(bar_drain);
    mbar_wait_drain(bar_drain, 0, wc, kSiteDrain);
  } else {
    const int hh = warp >> 2;                // query half of this warp's group
    const int r = (warp & 3) * 32 + lane;    // key row of the tile
    const int key = k0 + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int x0 = kHalfN * hh;
    bool ok = true;
    for (int st = 0; ok && st < nsteps; ++st) {
      const int ib = qb_lo + st % nq;
      const int q0 = ib * kBM;
      ok = mbar_wait_warp(bar_s_full(hh), st & 1u, wc, kSiteEw);
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
      auto vec4 = [&](int c, float (&l)[4], float (&d)[4]) {
        const float4 lv = ld_shared_v4f(vec + 4u * c);
        const float4 dv = ld_shared_v4f(vec + kBN * 4u + 4u * c);
        l[0] = lv.x; l[1] = lv.y; l[2] = lv.z; l[3] = lv.w;
        d[0] = dv.x; d[1] = dv.y; d[2] = dv.z; d[3] = dv.w;
      };
      uint32_t wpk[32], dspk[32];
      // two 32-column pieces (register pressure); the half is released after the second load
      auto pieces = [&](auto mtag) __attribute__((always_inline)) {
        constexpr bool kM = decltype(mtag)::value;
#pragma unroll
        for (int piece = 0; piece < 2; ++piece) {
          uint32_t xs[32], dxs[32];
          tmem_ld2_x32(tmem_base + lane_off + kColS + x0 + 32 * piece, xs,
                       tmem_base + lane_off + kColDP + x0 + 32 * piece, dxs);
          if (kSeparate && piece == 1) {
            tc_fence_before();
            mbar_arrive(bar_ld_free(hh));  // these columns may take the next step
          }
          elementwise_cols<32, BF16, true, kM>(xs, dxs, x0 + 32 * piece, p.c2, vis_lo, vis_hi, vec4,
                                               wpk + 16 * piece, dspk + 16 * piece);
        }
      };
      // warp-uniform choice: the pieces hold .sync.aligned TMEM loads, and the masked
      // path is exact for every lane
      if (__any_sync(0xffffffffu, masked))
        pieces(std::true_type{});
      else
        pieces(std::false_type{});
      // the single Pᵀ / dSᵀ buffer was read by step st - 1 (in place that is implied by
      // s_full; the wait keeps this thread at most one acc_done phase behind)
      if (st >= 1) {
        ok = mbar_wait_warp(bar_acc_done(hh, 0), (st - 1) & 1u, wc, kSiteEw);
        if (!ok) break;
        tc_fence_after();
      }
      tmem_st_x32(tmem_base + lane_off + kColPT + (kSeparate ? 32 * hh : kHalfN * hh), wpk);
      tmem_st_x32(tmem_base + lane_off + kColDST + (kSeparate ? 32 * hh : kHalfN * hh), dspk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p_full(hh, 0));
    }
    if (ok && nsteps > 0) {  // every MMA (both groups' shares) is complete
      ok = mbar_wait_warp(bar_drain, 0, wc, kSiteEw);
      if (ok) tc_fence_after();
    }
    const bool row_ok = key < p.L;
    const size_t off = ((static_cast<size_t>(b) * p.L + key) * p.Hkv + g) * D;
    if (ok && nsteps > 0) {  // group h writes columns [h D/2, (h + 1) D/2) of dK and dV
      store_acc_half<D, BF16, OUT_F32>(tmem_base + lane_off + kColDK, hh * (D / 2), p.scale, row_ok,
                                       p.dk, off);
      store_acc_half<D, BF16, OUT_F32>(tmem_base + lane_off + kColDV, hh * (D / 2), 1.f, row_ok,
                                       p.dv, off);
    }
    if (ok && nsteps == 0 && row_ok) {
      // no query sees these keys: zero gradients
      for (int c = hh * (D / 2); c < (hh + 1) * (D / 2); ++c) {
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
