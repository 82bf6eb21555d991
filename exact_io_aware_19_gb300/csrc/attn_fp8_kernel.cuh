// attn_fp8_kernel.cuh — exact attention forward on float8 e4m3 inputs, sm_103a.
//
// What it computes: the attention of the square kernels (same masks, GQA mapping,
// scale and LSE) on Q, K, V given as float8 e4m3, the FP8 path of the "Flash
// Attention optimization" skill page (workflow 3: inputs cast to float8_e4m3fn and
// run through FP8 attention kernels) and of "What is memory-efficient attention
// for long context on 8x H100?" (section 2: FlashAttention-3 adds FP8 support).
// Head dimension 64; O is written in bf16 or float32.
//
// Arithmetic: S = Q Kᵀ on the tensor cores (.kind::f8f6f4, fp32 accumulate, exact
// products of the e4m3 inputs). The softmax works in base 2 as in the other
// kernels; its weights are stored for the P·V MMA as e4m3 too, scaled to
// P' = 2^(x − m + 7) ≤ 256 so that they sit in e4m3's normal range, and the
// normaliser l' sums the same rounded P' values (the factor 2^7 cancels in O' / l').
// O' = Σ P'·V accumulates in fp32 in TMEM, and so does l': the B operand of the
// P·V MMA carries 16 rows of ones after the 64 rows of Vᵀ (N = 80), so O column 64
// is Σ P' summed by the tensor core from the very bytes it multiplies V with, and
// the O rescale scales it together with O.
//
// GB300 mapping (one CTA per 128-row tile, two CTAs per SM so that one CTA's
// softmax fills the other's waits; 256 TMEM columns and ~69 KiB of shared memory
// each):
//   * Q and K tiles: TMA boxes of 64 bytes (64 e4m3) per row, 64-byte swizzle.
//   * V is read as Vᵀ (keys contiguous), written by attn_fp8_transpose_v into the
//     workspace, so that both MMA operands are K-major: a 64 × 128-byte tile per
//     block, 128-byte swizzle, followed in its slot by the constant rows of ones.
//   * warp 4 (producer) streams K_j and Vᵀ_j into a ring of 10 KiB slots; warp 5
//     (MMA) issues S(j) into the TMEM S buffer, S(j + 1) as soon as the softmax
//     has read S(j) into registers (s_free), then O += P(j) Vᵀ(j) with P read
//     from TMEM (the A operand of a TS MMA: 8 columns of 4 e4m3 per K = 32).
//   * warps 0-3 (softmax): one thread per row; P' is converted to e4m3, packed four
//     keys to a 32-bit word and stored to the row's TMEM lane (32 columns) once the
//     P·V of the previous block, which read the one P' buffer, is done (pv_done;
//     s_full does not imply it, since S(j) is issued before P·V(j - 1)).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>
#include <type_traits>

#include "attn_kv_params.h"
#include "row_ops.cuh"
#include "sm103_ptx.cuh"
#include "tmem_io.cuh"

namespace ex19 {
namespace fp8 {

constexpr int kBM = 128;             // rows per tile (= TMEM lanes)
constexpr int kBN = 128;             // keys per block
constexpr int kD = 64;               // head dimension
constexpr int kThreads = 192;        // 4 softmax warps + producer warp + MMA warp
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kON = 80;              // P·V columns: O (64) and the normaliser (16 copies)
constexpr uint32_t kTmemCols = 256;  // S [0,128), O and l' [128, 208), P' [224, 256)
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;
constexpr uint32_t kColP = 224;      // P' of a block: 128 e4m3 per row, 4 per 32-bit column
constexpr int kPOffset = 7;          // P' = 2^(x - m + 7): at most 2^8 with the rescale threshold 1

enum : uint32_t {
  kSiteProdEmpty = 0xA0001,
  kSiteMmaQFull = 0xB0001, kSiteMmaKFull = 0xB0002, kSiteMmaVFull = 0xB0003,
  kSiteMmaPFull = 0xB0004, kSiteMmaDrain = 0xB0005,
  kSiteMmaSFree = 0xB0006,
  kSiteSmxSFull = 0xC0001, kSiteSmxOFull = 0xC0002, kSiteSmxPvDone = 0xC0003,
  kSiteDrainLoads = 0xD0001,
};

struct Fp8Geometry {
  static constexpr int kQBytes = kBM * kD;        // 8 KiB: 128 rows x 64 bytes
  static constexpr int kTileBytes = 8192;         // K_j (128 x 64 B) or Vᵀ_j (64 x 128 B)
  static constexpr int kOnesBytes = (kON - kD) * 128;  // rows of ones after Vᵀ_j
  static constexpr int kSlotBytes = kTileBytes + kOnesBytes;  // 10 KiB, 1 KiB aligned
  static constexpr int kSlots = 6;                // even: K_j in even slots, Vᵀ_j in odd
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = 8192;
  static constexpr int kOffBar = kOffKV + kSlots * kSlotBytes;
  // barriers: full[S], empty[S], q_full, s_full, s_free, p_full[2], pv_done[2], o_full, drain
  static constexpr int kNumBars = 2 * kSlots + 9;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemUsed = kOffMisc + 16;
  static constexpr int kSmemBytes = kSmemUsed + 1024;
};

// Two e4m3 values of two fp32 weights (low byte: the first), rounded to nearest.
__device__ __forceinline__ uint32_t e4m3x2_of_f32(float first, float second) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
  return static_cast<uint32_t>(r);
}

template <bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 2)
    attn_fp8_sm103_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_vt, const KvParams p) {
  using G = Fp8Geometry;
  constexpr int S = G::kSlots;
  // move the reference max when a score exceeds it by more than 2^1: P' stays at most
  // 2^(1 + kPOffset) = 256, inside e4m3's range (448)
  constexpr float kThresh = 1.0f;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + G::kOffQ;
  const uint32_t sKV = sbase + G::kOffKV;
  const uint32_t bars = sbase + G::kOffBar;
  auto bar_full = [&](uint32_t s) { return bars + 8u * s; };
  auto bar_empty = [&](uint32_t s) { return bars + 8u * (S + s); };
  const uint32_t bar_q_full = bars + 8u * (2 * S);
  const uint32_t bar_s_full = bars + 8u * (2 * S + 1);
  const uint32_t bar_s_free = bars + 8u * (2 * S + 2);
  auto bar_p_full = [&](uint32_t b) { return bars + 8u * (2 * S + 3 + b); };
  auto bar_pv_done = [&](uint32_t b) { return bars + 8u * (2 * S + 5 + b); };
  const uint32_t bar_o_full = bars + 8u * (2 * S + 7);
  const uint32_t bar_drain = bars + 8u * (2 * S + 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + G::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: (batch, K/V head, 128-row tile); the group's query heads share the tile.
  int x = blockIdx.x;
  const int rt = x % p.row_tiles;
  x /= p.row_tiles;
  const int g = x % p.Hkv;
  const int b = x / p.Hkv;
  const int i0 = rt * p.q_per_tile, i1 = min(p.Lq, i0 + p.q_per_tile);
  const int L = p.Lk;
  const int nblk = (L + kBN - 1) / kBN;
  const int wr = p.causal ? 0 : p.window_right;
  const int blk_hi = (wr >= 0) ? min(nblk, (i1 - 1 + wr) / kBN + 1) : nblk;
  const int blk_lo = (p.window_left >= 0) ? max(0, i0 - p.window_left) / kBN : 0;
  const int nblocks = max(0, blk_hi - blk_lo);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_q_full, 1);
    mbar_init(bar_s_full, 1);
    mbar_init(bar_s_free, kBM);
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar_p_full(k), kBM);
      mbar_init(bar_pv_done(k), 1);
    }
    mbar_init(bar_o_full, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_vt);
  }
  // Launched as a programmatic dependent of the V transpose: past this point Vᵀ (and
  // everything before it on the stream) is complete and visible. TMEM is allocated
  // only after it, so this CTA never holds TMEM while it waits on another kernel.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  // the rows of ones (e4m3 1.0 = 0x38) behind every slot's tile; the TMA loads never
  // write them
  for (int t = threadIdx.x; t < S * (G::kOnesBytes / 16); t += kThreads) {
    const int slot = t / (G::kOnesBytes / 16), c = t % (G::kOnesBytes / 16);
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(
                     sKV + slot * G::kSlotBytes + G::kTileBytes + c * 16),
                 "r"(0x38383838u)
                 : "memory");
  }
  fence_proxy_async_shared();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  WaitCtl wc;
  wc.abort_flag = abort_flag;
  wc.status = p.status;
  wc.set_limit(p.wait_limit_ns);
  wc.unit = blockIdx.x;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && nblocks > 0) {
      mbar_arrive_expect_tx(bar_q_full, 64u * p.group * p.q_per_tile);
      tma_load_4d(sQ, &tm_q, bar_q_full, 0, g * p.group, i0, b);
      uint32_t n = 0;
      bool ok = true;
      for (int j = blk_lo; ok && j < blk_hi; ++j) {
        for (int kv = 0; kv < 2; ++kv) {
          const uint32_t slot = n % S;
          ok = mbar_wait_bounded(bar_empty(slot), ((n / S) & 1u) ^ 1u, wc, kSiteProdEmpty);
          if (!ok) break;
          mbar_arrive_expect_tx(bar_full(slot), G::kTileBytes);
          if (kv == 0)  // K_j: 128 keys x 64 bytes
            tma_load_4d(sKV + slot * G::kSlotBytes, &tm_k, bar_full(slot), 0, g, j * kBN, b);
          else  // Vᵀ_j: 64 rows (d) x 128 bytes (keys)
            tma_load_4d(sKV + slot * G::kSlotBytes, &tm_vt, bar_full(slot), j * kBN, 0, g, b);
          ++n;
        }
      }
      // Whether or not this CTA aborted, the copies issued last may still be in
      // flight (another role can abort after this loop has ended, and then nothing
      // consumes them): let them land before the CTA can exit.
      {
        for (uint32_t back = 1; back <= S && back <= n; ++back) {
          const uint32_t m = n - back;
          mbar_wait_drain(bar_full(m % S), (m / S) & 1u, wc, kSiteDrainLoads);
        }
        mbar_wait_drain(bar_q_full, 0, wc, kSiteDrainLoads);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA issuer
    if (nblocks > 0) {
      constexpr uint32_t idesc_s = idesc_f16_f32acc(false, kBM, kBN, false);  // e4m3 x e4m3
      constexpr uint32_t idesc_o = idesc_f16_f32acc(false, kBM, kON, false);
      const uint64_t dq = sdesc_swizzled(sQ, 16, 512, 4);      // 64-byte rows, 64-byte swizzle
      const uint64_t dk = sdesc_swizzled(sKV, 16, 512, 4);
      const uint64_t dvt = sdesc_swizzled(sKV, 16, 1024, 2);   // 128-byte rows, 128-byte swizzle
      const uint32_t mO = tmem_base + kColO;
      auto slot_of = [&](uint32_t idx) { return idx % S; };
      auto par_of = [&](uint32_t idx) { return (idx / S) & 1u; };
      // S = Q · K_jᵀ into the TMEM S buffer (two MMAs of K = 32 bytes); releases K_j.
      auto issue_s = [&](int jj) __attribute__((always_inline)) -> bool {
        const uint32_t kidx = 2u * jj;
        if (!mbar_wait_warp(bar_full(slot_of(kidx)), par_of(kidx), wc, kSiteMmaKFull)) return false;
        tc_fence_after();
        const uint32_t mS = tmem_base + kColS;
        const uint64_t dks = dk + ((slot_of(kidx) * G::kSlotBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kD / 32; ++kk)
          mma_ss_f8_elect(mS, dq + (kk * 32 >> 4), dks + (kk * 32 >> 4), idesc_s, kk > 0 ? 1u : 0u);
        mma_commit_elect(bar_s_full);
        mma_commit_elect(bar_empty(slot_of(kidx)));
        return true;
      };
      // [O | l'] (+)= P(jj) · [V_j | 1] with P from TMEM (8 columns per MMA of K = 32
      // keys) and Vᵀ_j and the ones from its slot (four MMAs); releases Vᵀ_j.
      auto issue_pv = [&](int jj) __attribute__((always_inline)) -> bool {
        const uint32_t vidx = 2u * jj + 1u;
        if (!mbar_wait_warp(bar_full(slot_of(vidx)), par_of(vidx), wc, kSiteMmaVFull)) return false;
        if (!mbar_wait_warp(bar_p_full(jj & 1), (jj >> 1) & 1u, wc, kSiteMmaPFull)) return false;
        tc_fence_after();
        const uint64_t dvs = dvt + ((slot_of(vidx) * G::kSlotBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBN / 32; ++kk)
          mma_ts_f8_elect(mO, tmem_base + kColP + 8 * kk, dvs + (kk * 32 >> 4), idesc_o,
                          (jj == 0 && kk == 0) ? 0u : 1u);
        mma_commit_elect(bar_pv_done(jj & 1));
        mma_commit_elect(bar_empty(slot_of(vidx)));
        return true;
      };
      bool ok = mbar_wait_warp(bar_q_full, 0, wc, kSiteMmaQFull);
      if (ok) {
        tc_fence_after();
        ok = issue_s(0);
        for (int jj = 0; ok && jj < nblocks; ++jj) {
          if (jj + 1 < nblocks) {  // S(jj + 1) once the softmax holds S(jj) in registers
            ok = mbar_wait_warp(bar_s_free, jj & 1u, wc, kSiteMmaSFree);
            if (ok) {
              tc_fence_after();
              ok = issue_s(jj + 1);
            }
          }
          if (ok) ok = issue_pv(jj);
        }
        if (ok) mma_commit_elect(bar_o_full);
      }
    }
    mma_commit_elect(bar_drain);
    mbar_wait_drain(bar_drain, 0, wc, kSiteMmaDrain);
  } else {
    // -------------------------------------------------------- softmax warps
    const int rho = warp * 32 + lane;  // row of the tile
    const bool row_ok = rho < (i1 - i0) * p.group;
    const int qi = i0 + rho / p.group;
    const int h = g * p.group + rho % p.group;
    const int pos_min = i0, pos_max = i1 - 1;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tO = tmem_base + lane_off + kColO;
    const float C = p.score_log2;
    const bool neg = p.negate_scores != 0;
    const float Cs = neg ? -C : C;
    float m_ref = -INFINITY;  // reference max (base-2 units)
    bool ok = true;
    // One key block (jj-th of this CTA); false when a wait gave up. Blocks that cross
    // a mask boundary run the masked instantiation outside the unmasked middle's own
    // tight loop, so the hot loop holds one block body only.
    auto one_block = [&](int jj, auto masked_tag) __attribute__((always_inline)) -> bool {
      constexpr bool masked = decltype(masked_tag)::value;
      const int j = blk_lo + jj;
      const uint32_t buf = jj & 1;
      if (!mbar_wait_warp(bar_s_full, jj & 1u, wc, kSiteSmxSFull)) return false;
      tc_fence_after();
      const uint32_t tS = tmem_base + lane_off + kColS;
      const int key0 = j * kBN;
      int vis_lo = 0, vis_hi = kBN;
      if constexpr (masked) {
        const int hi_key = (wr >= 0) ? min(L, qi + wr + 1) : L;
        const int lo_key = (p.window_left >= 0) ? qi - p.window_left : 0;
        vis_hi = max(0, min(kBN, hi_key - key0));
        vis_lo = max(0, min(kBN, lo_key - key0));
      }
      float alpha = 1.f;
      bool rescale = false;
      bool stop = false;
      auto block_body = [&](auto masked_tag) __attribute__((always_inline)) {
        constexpr bool M = decltype(masked_tag)::value;
        uint32_t sr[128];
        tmem_ld_x128(tS, sr);
        tc_fence_before();
        mbar_arrive(bar_s_free);  // the S buffer may take S(jj + 1)
        if constexpr (M) {
          const uint32_t fill = neg ? 0x7f800000u : 0xff800000u;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c < vis_lo || c >= vis_hi) sr[c] = fill;
        }
        float mx;
        {
          float sv[128];
#pragma unroll
          for (int c = 0; c < 128; ++c) sv[c] = __uint_as_float(sr[c]);
          mx = neg ? -row_min128(sv) : row_max128(sv);
        }
        const float bm = (mx == -INFINITY) ? -INFINITY : mx * C;
        if (bm > m_ref + kThresh) {
          alpha = ex2_approx(m_ref - bm);
          m_ref = bm;
          rescale = true;
        }
        // x - m + 7 with the reference max of this block
        const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
        const float nmu = static_cast<float>(kPOffset) - mu;
        // The one P' buffer was read by P·V(jj - 1) (issued after S(jj), so s_full
        // does not cover it): wait until that MMA is done before storing P'(jj).
        if (jj >= 1) {
          if (!mbar_wait_warp(bar_pv_done((jj - 1) & 1), ((jj - 1) >> 1) & 1u, wc, kSiteSmxPvDone)) {
            stop = true;
            return;
          }
          tc_fence_after();
        }
        // P' of the row to its TMEM lane: key k in byte k mod 4 of column k / 4, stored
        // 32 keys (8 columns) at a time so that few words are live at once.
#pragma unroll
        for (int q32 = 0; q32 < 4; ++q32) {
          uint32_t w[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {  // 4 keys per 32-bit word
            uint32_t e2[2];
#pragma unroll
            for (int v2 = 0; v2 < 2; ++v2) {
              const int c = q32 * 32 + u * 4 + v2 * 2;
              const float2 xx = __ffma2_rn(
                  make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])),
                  make_float2(Cs, Cs), make_float2(nmu, nmu));
              // fp32 exponentials and one conversion per pair (converting the
              // arguments to fp16 pairs for a packed exponential measured slower: a
              // second conversion on the ALU pipe, the busiest one here)
              float p0 = ex2_approx(xx.x), p1 = ex2_approx(xx.y);
              if constexpr (M) {  // masked keys get exactly 0
                p0 = (c >= vis_lo && c < vis_hi) ? p0 : 0.f;
                p1 = (c + 1 >= vis_lo && c + 1 < vis_hi) ? p1 : 0.f;
              }
              e2[v2] = e4m3x2_of_f32(p0, p1);
            }
            w[u] = e2[0] | (e2[1] << 16);
          }
          tmem_st_x8(tmem_base + lane_off + kColP + 8 * q32, w);
        }
        tmem_st_wait();
      };
      block_body(masked_tag);
      if (stop) return false;
      // O rescale once the previous P·V is complete; the first block's P·V overwrites O.
      if (__any_sync(0xffffffffu, rescale && jj > 0)) {
        if (!mbar_wait_warp(bar_pv_done((jj - 1) & 1), ((jj - 1) >> 1) & 1u, wc, kSiteSmxPvDone))
          return false;
        tc_fence_after();
        const float a = (rescale && jj > 0) ? alpha : 1.f;
#pragma unroll
        for (int c0 = 0; c0 < kD; c0 += 32) {
          uint32_t orow[32];
          tmem_ld_x32(tO + c0, orow);
#pragma unroll
          for (int c = 0; c < 32; ++c) orow[c] = __float_as_uint(__uint_as_float(orow[c]) * a);
          tmem_st_x32(tO + c0, orow);
        }
        {  // l' (column 64; its 15 copies are never read)
          uint32_t lrow[16];
          tmem_ld_x16(tO + kD, lrow);
#pragma unroll
          for (int c = 0; c < 16; ++c) lrow[c] = __float_as_uint(__uint_as_float(lrow[c]) * a);
          tmem_st_x16(tO + kD, lrow);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar_p_full(buf));
      return true;
    };
    {
      // Blocks [ja, jb) of this CTA cross no mask boundary (the one-tile kernel's rule).
      int ja = 0, jb = nblocks;
      if (p.window_left >= 0) {  // key0 >= pos_max - window_left
        const int first = pos_max - p.window_left;
        if (first > 0) ja = max(ja, (first + kBN - 1) / kBN - blk_lo);
      }
      jb = min(jb, L / kBN - blk_lo);  // key0 + kBN <= L
      if (wr >= 0) {                   // key0 + kBN - 1 <= pos_min + wr
        const int last = pos_min + wr - (kBN - 1);
        jb = min(jb, last >= 0 ? last / kBN + 1 - blk_lo : 0);
      }
      ja = min(max(ja, 0), nblocks);
      jb = max(jb, ja);
      for (int jj = 0; ok && jj < nblocks;) {
        if (jj >= ja && jj < jb) {
          for (; ok && jj < jb; ++jj) ok = one_block(jj, std::false_type{});
        } else {
          ok = one_block(jj, std::true_type{});
          ++jj;
        }
      }
    }
    if (ok && nblocks > 0) {
      ok = mbar_wait_warp(bar_o_full, 0, wc, kSiteSmxOFull);
      if (ok) tc_fence_after();
    }
    if (ok && nblocks > 0) {
      float l;
      {
        uint32_t lrow[16];
        tmem_ld_x16(tO + kD, lrow);
        l = __uint_as_float(lrow[0]);
      }
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const size_t orow_off = ((static_cast<size_t>(b) * p.Lq + qi) * p.Hq + h) * kD;
#pragma unroll
      for (int c0 = 0; c0 < kD; c0 += 32) {
        uint32_t orow[32];
        tmem_ld_x32(tO + c0, orow);
        if (!row_ok) continue;
        if constexpr (OUT_F32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow_off + c0);
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            dst[c >> 2] = make_float4(__uint_as_float(orow[c]) * inv_l,
                                      __uint_as_float(orow[c + 1]) * inv_l,
                                      __uint_as_float(orow[c + 2]) * inv_l,
                                      __uint_as_float(orow[c + 3]) * inv_l);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + orow_off + c0);
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint4 wv;
            wv.x = pack2(__uint_as_float(orow[c]) * inv_l, __uint_as_float(orow[c + 1]) * inv_l, true);
            wv.y = pack2(__uint_as_float(orow[c + 2]) * inv_l, __uint_as_float(orow[c + 3]) * inv_l, true);
            wv.z = pack2(__uint_as_float(orow[c + 4]) * inv_l, __uint_as_float(orow[c + 5]) * inv_l, true);
            wv.w = pack2(__uint_as_float(orow[c + 6]) * inv_l, __uint_as_float(orow[c + 7]) * inv_l, true);
            dst[c >> 3] = wv;
          }
        }
      }
      if (row_ok && p.lse != nullptr) {
        const float lse2 = (l > 0.f) ? m_ref - static_cast<float>(kPOffset) + lg2_approx(l) : -INFINITY;
        p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.Lq + qi] =
            (l > 0.f) ? lse2 * 0.69314718055994531f : -INFINITY;
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Vᵀ for the P·V MMA: v [B, L, Hkv, 64] e4m3 -> vt [B, Hkv, 64, Lp] (keys contiguous,
// Lp = L rounded up to 16; keys L .. Lp-1 are zero). One CTA of 4 warps per (128 keys,
// head, batch): warp w moves bytes 16w .. 16w + 15 of d, lane l keys 4l .. 4l + 3.
// A lane loads its 4 keys' 16-byte pieces, transposes each 4 x 4 byte block in
// registers (byte permutes) and stores 16 words, one per d row: the warp's 32 lanes
// write 128 consecutive bytes of that row.
__global__ void __launch_bounds__(128) attn_fp8_transpose_v(const uint8_t* __restrict__ v,
                                                            uint8_t* __restrict__ vt, int L,
                                                            int Hkv, int Lp) {
  const int g = blockIdx.y, b = blockIdx.z;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = blockIdx.x * 128 + 4 * lane;  // first key of this lane (Lp is a multiple of 4)
  if (k >= Lp) return;
  uint32_t a[4][4];  // a[i][q]: bytes 16w + 4q .. + 3 of key k + i
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (k + i < L)
      val = *reinterpret_cast<const uint4*>(v + ((static_cast<size_t>(b) * L + k + i) * Hkv + g) * 64 + 16 * w);
    a[i][0] = val.x;
    a[i][1] = val.y;
    a[i][2] = val.z;
    a[i][3] = val.w;
  }
  uint8_t* dst = vt + ((static_cast<size_t>(b) * Hkv + g) * 64 + 16 * w) * Lp + k;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    // 4 x 4 byte transpose: t0 .. t3 pair up the keys' bytes, col[e] = byte e of keys 0 .. 3
    const uint32_t t0 = __byte_perm(a[0][q], a[1][q], 0x5140);  // k0.b0 k1.b0 k0.b1 k1.b1
    const uint32_t t1 = __byte_perm(a[2][q], a[3][q], 0x5140);  // k2.b0 k3.b0 k2.b1 k3.b1
    const uint32_t t2 = __byte_perm(a[0][q], a[1][q], 0x7362);  // k0.b2 k1.b2 k0.b3 k1.b3
    const uint32_t t3 = __byte_perm(a[2][q], a[3][q], 0x7362);  // k2.b2 k3.b2 k2.b3 k3.b3
    const uint32_t col[4] = {__byte_perm(t0, t1, 0x5410), __byte_perm(t0, t1, 0x7632),
                             __byte_perm(t2, t3, 0x5410), __byte_perm(t2, t3, 0x7632)};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      *reinterpret_cast<uint32_t*>(dst + static_cast<size_t>(4 * q + e) * Lp) = col[e];
  }
}

}  // namespace fp8
}  // namespace ex19
