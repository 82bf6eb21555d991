// attn_fwd_kernel.cuh — exact attention forward for sm_103a (GB300).
//
// What it computes: O = softmax(scale · Q Kᵀ + mask) V and the per-row
// log-sum-exp, the standard attention of the "Flash Attention optimization" skill
// page (workflow 1 step 2; workflow 2 steps 2-3 for causal, MQA/GQA and the
// window), evaluated the IO-aware way of "What is memory-efficient attention for
// long context on 8x H100?" section 2: blocks of Q, K, V are staged on chip, the
// softmax is accumulated online (running max and running sum), and only O and LSE
// are written back, so the L x L score matrix never reaches HBM.
//
// GB300 mapping (one CTA per SM, persistent):
//   * A work unit is 256 query rows of one (batch, head): two 128-row tiles that
//     share one stream of K/V blocks of 128 keys.
//   * warp 8   (producer): TMA loads of the Q tiles and of K_j, V_j into a ring of
//              shared-memory slots (128-byte swizzle), signalled by mbarriers.
//   * warp 9   (MMA): one thread issues tcgen05.mma. S_t = Q_t K_jᵀ goes to TMEM
//              (fp32, 128 columns per tile); O_t += P_t V_j reads P_t from TMEM
//              (16-bit, aliased over S_t) and V_j from shared memory. MMAs of the
//              two tiles are interleaved so one tile's softmax overlaps the other
//              tile's MMAs.
//   * warps 0-3 / 4-7 (softmax, tile 0 / tile 1): one thread per query row (TMEM
//              lane). Loads its row of S, masks boundary blocks, keeps the running
//              max m (base-2 units) and sum l, writes P = 2^(x - m) back to TMEM,
//              rescales its O row when m grows by more than 2^8, and at the end of
//              the unit writes O / l and LSE.
//   * Every wait is bounded (globaltimer); a wait that runs out records a timeout
//     in the status word and every role leaves its loop, so the CTA still frees
//     its TMEM and exits.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "attn_params.h"
#include "sm103_ptx.cuh"
#include "tmem_io.cuh"

namespace ex19 {

constexpr int kBM = 128;             // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;             // keys per K/V block
constexpr int kTilesPerUnit = 2;     // query tiles per work unit
constexpr int kUnitRows = kBM * kTilesPerUnit;
constexpr int kThreads = 320;        // 8 softmax warps + producer warp + MMA warp
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;  // S0 [0,128) S1 [128,256) O0 [256,..) O1 [384,..)
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when m grows > 2^8

// Wait sites (for the status word): role << 16 | site
enum : uint32_t {
  kSiteProdEmpty = 0x10001, kSiteProdQFree = 0x10002,
  kSiteMmaQFull = 0x20001, kSiteMmaKFull = 0x20002, kSiteMmaVFull = 0x20003,
  kSiteMmaPFull = 0x20004, kSiteMmaOFree = 0x20005, kSiteMmaDrain = 0x20006,
  kSiteSmxSFull = 0x30001, kSiteSmxOFull = 0x30002,
  kSiteDrainLoads = 0x40001,
};

template <int D>
struct Geometry {
  static constexpr int kChunks = D / 64;          // 64-element (128-byte) swizzle boxes per row
  static constexpr int kChunkBytes = kBM * 128;   // 128 rows x 128 bytes
  static constexpr int kTileBytes = kBM * D * 2;  // one 128-row tile of Q, K or V
  static constexpr int kSlots = (D == 64) ? 8 : 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kTilesPerUnit * kTileBytes;
  static constexpr int kOffBar = kOffKV + kSlots * kTileBytes;
  // barriers: full[S], empty[S], q_full, q_free, s_full[2], p_full[2], o_full[2], o_free[2], drain
  static constexpr int kNumBars = 2 * kSlots + 11;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kSmemUsed = kOffMisc + 16;
  static constexpr int kSmemBytes = kSmemUsed + 1024;     // slack to align the base to 1024
};

// Rows and key blocks of one query tile of a unit.
struct TileSpan {
  int row0;    // first query row
  int lo, hi;  // key blocks [lo, hi) this tile visits (empty when lo >= hi)
};

struct Unit {
  int b, h, g;
  TileSpan t[kTilesPerUnit];
  int lo, hi;  // union of the tiles' block ranges
};

__device__ __forceinline__ TileSpan tile_span(const FwdParams& p, int row0) {
  TileSpan s;
  s.row0 = row0;
  if (row0 >= p.L) {
    s.lo = 0;
    s.hi = 0;
    return s;
  }
  const int last = min(row0 + kBM - 1, p.L - 1);
  const int nblk = (p.L + kBN - 1) / kBN;
  s.hi = p.causal ? (last / kBN + 1) : nblk;
  s.lo = (p.window_left >= 0) ? max(0, row0 - p.window_left) / kBN : 0;
  return s;
}

// k-th unit of this CTA. Ranks are dealt to CTAs in a snake order over a
// heavy-first ranking (causal: the last row blocks see the most keys).
__device__ __forceinline__ bool unit_of(const FwdParams& p, int k, Unit& u) {
  const int G = gridDim.x;
  const int c = blockIdx.x;
  const long long r = static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - c) : c);
  if (r >= p.num_units) return false;
  const int BH = p.B * p.Hq;
  const int mb = p.units_per_bh - 1 - static_cast<int>(r / BH);
  const int bh = static_cast<int>(r % BH);
  u.b = bh / p.Hq;
  u.h = bh % p.Hq;
  u.g = u.h / (p.Hq / p.Hkv);
  u.lo = 0x7fffffff;
  u.hi = 0;
  for (int t = 0; t < kTilesPerUnit; ++t) {
    u.t[t] = tile_span(p, mb * kUnitRows + t * kBM);
    if (u.t[t].lo < u.t[t].hi) {
      u.lo = min(u.lo, u.t[t].lo);
      u.hi = max(u.hi, u.t[t].hi);
    }
  }
  return true;
}

__device__ __forceinline__ bool has_block(const TileSpan& s, int j) { return j >= s.lo && j < s.hi; }

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

template <int D, bool BF16, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_sm103_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using G = Geometry<D>;
  constexpr int S = G::kSlots;
  // bf16 P is split into hi + lo halves (two P·V MMAs) so that rounding P to 8
  // significant bits does not dominate the output error; fp16 P has 11 bits.
  constexpr bool kSplitP = BF16;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + G::kOffQ;
  const uint32_t sKV = sbase + G::kOffKV;
  const uint32_t bars = sbase + G::kOffBar;
  auto bar_full = [&](int s) { return bars + 8u * s; };
  auto bar_empty = [&](int s) { return bars + 8u * (S + s); };
  const uint32_t bar_q_full = bars + 8u * (2 * S);
  const uint32_t bar_q_free = bars + 8u * (2 * S + 1);
  auto bar_s_full = [&](int t) { return bars + 8u * (2 * S + 2 + t); };
  auto bar_p_full = [&](int t) { return bars + 8u * (2 * S + 4 + t); };
  auto bar_o_full = [&](int t) { return bars + 8u * (2 * S + 6 + t); };
  auto bar_o_free = [&](int t) { return bars + 8u * (2 * S + 8 + t); };
  const uint32_t bar_drain = bars + 8u * (2 * S + 10);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + G::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_q_full, 1);
    mbar_init(bar_q_free, 1);
    for (int t = 0; t < kTilesPerUnit; ++t) {
      mbar_init(bar_s_full(t), 1);
      mbar_init(bar_p_full(t), kBM);
      mbar_init(bar_o_full(t), 1);
      mbar_init(bar_o_free(t), kBM);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  WaitCtl wc;
  wc.abort_flag = abort_flag;
  wc.status = p.status;
  wc.limit_ns = p.wait_limit_ns;
  wc.unit = 0;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;      // K/V slot loads issued
      uint32_t q_cnt = 0;   // Q loads issued
      bool ok = true;
      Unit u;
      for (int k = 0; ok && unit_of(p, k, u); ++k) {
        wc.unit = k;
        ok = mbar_wait_bounded(bar_q_free, (q_cnt & 1u) ^ 1u, wc, kSiteProdQFree);
        if (!ok) break;
        uint32_t qbytes = 0;
        for (int t = 0; t < kTilesPerUnit; ++t)
          if (u.t[t].lo < u.t[t].hi) qbytes += G::kTileBytes;
        mbar_arrive_expect_tx(bar_q_full, qbytes);
        for (int t = 0; t < kTilesPerUnit; ++t) {
          if (u.t[t].lo >= u.t[t].hi) continue;
          for (int c = 0; c < G::kChunks; ++c)
            tma_load_4d(sQ + t * G::kTileBytes + c * G::kChunkBytes, &tm_q, bar_q_full, c * 64,
                        u.h, u.t[t].row0, u.b);
        }
        ++q_cnt;
        for (int j = u.lo; ok && j < u.hi; ++j) {
          for (int kv = 0; kv < 2; ++kv) {
            const uint32_t slot = it % S;
            ok = mbar_wait_bounded(bar_empty(slot), ((it / S) & 1u) ^ 1u, wc, kSiteProdEmpty);
            if (!ok) break;
            mbar_arrive_expect_tx(bar_full(slot), G::kTileBytes);
            const CUtensorMap* tm = kv ? &tm_v : &tm_k;
            for (int c = 0; c < G::kChunks; ++c)
              tma_load_4d(sKV + slot * G::kTileBytes + c * G::kChunkBytes, tm, bar_full(slot),
                          c * 64, u.g, j * kBN, u.b);
            ++it;
          }
        }
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA can exit.
        for (uint32_t back = 1; back <= S && back <= it; ++back) {
          const uint32_t n = it - back;
          mbar_wait_drain(bar_full(n % S), (n / S) & 1u, wc, kSiteDrainLoads);
        }
        if (q_cnt > 0) mbar_wait_drain(bar_q_full, (q_cnt - 1) & 1u, wc, kSiteDrainLoads);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16_f32acc(BF16, kBM, kBN, false);
      constexpr uint32_t idesc_o = idesc_f16_f32acc(BF16, kBM, D, true);
      uint32_t it = 0, q_cnt = 0;
      uint32_t p_cnt[kTilesPerUnit] = {0, 0};
      uint32_t o_cnt[kTilesPerUnit] = {0, 0};
      bool ok = true;
      Unit u;
      for (int k = 0; ok && unit_of(p, k, u); ++k) {
        wc.unit = k;
        ok = mbar_wait_bounded(bar_q_full, q_cnt & 1u, wc, kSiteMmaQFull);
        ++q_cnt;
        if (!ok) break;
        tc_fence_after();
        int pend[kTilesPerUnit] = {-1, -1};          // block whose S_t waits for its P·V
        uint32_t pend_vslot[kTilesPerUnit] = {0, 0};
        uint32_t pend_vpar[kTilesPerUnit] = {0, 0};
        bool first_pv[kTilesPerUnit] = {true, true};
        uint32_t prev_vslot = 0;
        bool have_prev_v = false;

        // O_t (+)= P_t · V for the pending block of tile t.
        auto issue_pv = [&](int t) -> bool {
          if (!mbar_wait_bounded(bar_full(pend_vslot[t]), pend_vpar[t], wc, kSiteMmaVFull))
            return false;
          if (!mbar_wait_bounded(bar_p_full(t), p_cnt[t] & 1u, wc, kSiteMmaPFull)) return false;
          ++p_cnt[t];
          if (first_pv[t]) {
            if (!mbar_wait_bounded(bar_o_free(t), (o_cnt[t] & 1u) ^ 1u, wc, kSiteMmaOFree))
              return false;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + 256 + 128 * t;
          const uint32_t p_tmem = tmem_base + 128 * t;
          const uint32_t v_addr = sKV + pend_vslot[t] * G::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            // 16 keys per MMA: 8 TMEM columns of packed P, 16 rows (2 KiB) of V.
            const uint64_t bdesc = sdesc_sw128(v_addr + kk * 2048, G::kChunkBytes, 1024);
            mma_ts(d_tmem, p_tmem + kk * 8, bdesc, idesc_o, (first_pv[t] && kk == 0) ? 0u : 1u);
          }
          if (kSplitP) {
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk) {
              const uint64_t bdesc = sdesc_sw128(v_addr + kk * 2048, G::kChunkBytes, 1024);
              mma_ts(d_tmem, p_tmem + 64 + kk * 8, bdesc, idesc_o, 1u);
            }
          }
          first_pv[t] = false;
          pend[t] = -1;
          return true;
        };

        for (int j = u.lo; ok && j < u.hi; ++j) {
          const uint32_t kslot = it % S, kpar = (it / S) & 1u;
          ++it;
          const uint32_t vslot = it % S, vpar = (it / S) & 1u;
          ++it;
          ok = mbar_wait_bounded(bar_full(kslot), kpar, wc, kSiteMmaKFull);
          if (!ok) break;
          tc_fence_after();
          for (int t = 0; t < kTilesPerUnit; ++t) {
            const bool flushed = pend[t] >= 0;
            if (flushed && !(ok = issue_pv(t))) break;
            if (has_block(u.t[t], j)) {
              // S_t = Q_t · K_jᵀ  (D/16 MMAs of K = 16)
              const uint32_t q_addr = sQ + t * G::kTileBytes;
              const uint32_t k_addr = sKV + kslot * G::kTileBytes;
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * G::kChunkBytes + (kk & 3) * 32;
                mma_ss(tmem_base + 128 * t, sdesc_sw128(q_addr + off, 16, 1024),
                       sdesc_sw128(k_addr + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
              }
              mma_commit(bar_s_full(t));
              pend[t] = j;
              pend_vslot[t] = vslot;
              pend_vpar[t] = vpar;
            } else if (flushed) {
              mma_commit(bar_o_full(t));  // that was tile t's last block
              ++o_cnt[t];
            }
          }
          if (!ok) break;
          mma_commit(bar_empty(kslot));
          if (have_prev_v) mma_commit(bar_empty(prev_vslot));
          prev_vslot = vslot;
          have_prev_v = true;
        }
        for (int t = 0; ok && t < kTilesPerUnit; ++t) {
          if (pend[t] >= 0) {
            if (!(ok = issue_pv(t))) break;
            mma_commit(bar_o_full(t));
            ++o_cnt[t];
          }
        }
        if (!ok) break;
        if (have_prev_v) mma_commit(bar_empty(prev_vslot));
        mma_commit(bar_q_free);
      }
      // Every MMA this thread issued has finished once the drain barrier flips.
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0, wc, kSiteMmaDrain);
    }
  } else {
    // -------------------------------------------------------- softmax warps
    const int t = warp >> 2;
    const int quarter = warp & 3;
    const int r_in_tile = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem_base + lane_off + 128 * t;
    const uint32_t tO = tmem_base + lane_off + 256 + 128 * t;
    const float C = p.score_log2;
    uint32_t s_cnt = 0, o_cnt = 0;
    bool ok = true;
    Unit u;
    for (int k = 0; ok && unit_of(p, k, u); ++k) {
      wc.unit = k;
      const TileSpan span = u.t[t];
      if (span.lo >= span.hi) continue;
      const int row = span.row0 + r_in_tile;
      float m_ref = -INFINITY;  // reference max (base-2 units) the P values are relative to
      float l = 0.f;            // running sum of P
      for (int j = span.lo; j < span.hi; ++j) {
        ok = mbar_wait_warp(bar_s_full(t), s_cnt & 1u, wc, kSiteSmxSFull);
        ++s_cnt;
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld_x128(tS, sr);
        float s[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
        if (p.negate_scores) {
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = -s[c];
        }
        const int key0 = j * kBN;
        const bool masked = (key0 + kBN > p.L) || (p.causal && key0 + kBN - 1 > span.row0) ||
                            (p.window_left >= 0 && key0 < span.row0 + kBM - 1 - p.window_left);
        int vis_lo = 0, vis_hi = kBN;  // visible columns of this row: [vis_lo, vis_hi)
        if (masked) {
          int hi_key = p.L;
          if (p.causal) hi_key = min(hi_key, row + 1);
          int lo_key = (p.window_left >= 0) ? row - p.window_left : 0;
          vis_hi = max(0, min(kBN, hi_key - key0));
          vis_lo = max(0, min(kBN, lo_key - key0));
        }
        float mx = -INFINITY;
        if (!masked) {
#pragma unroll
          for (int c = 0; c < 128; ++c) mx = fmaxf(mx, s[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= vis_lo && c < vis_hi) mx = fmaxf(mx, s[c]);
        }
        const float bm = (mx == -INFINITY) ? -INFINITY : mx * C;
        float alpha = 1.f;
        bool rescale = false;
        if (bm > m_ref + kRescaleThreshold) {
          alpha = ex2_approx(m_ref - bm);  // 0 when m_ref is -inf
          m_ref = bm;
          rescale = true;
        }
        const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
        float sum0 = 0.f, sum1 = 0.f;
        // P in 32-column chunks: 16 packed registers per chunk, stored to TMEM
        // over the S columns already read (P hi at column c/2, P lo at 64 + c/2).
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t pk[16];
          uint32_t pk_lo[16];
#pragma unroll
          for (int c = c0; c < c0 + 32; c += 2) {
            float p0 = ex2_approx(fmaf(s[c], C, -mu));
            float p1 = ex2_approx(fmaf(s[c + 1], C, -mu));
            if (masked) {
              p0 = (c >= vis_lo && c < vis_hi) ? p0 : 0.f;
              p1 = (c + 1 >= vis_lo && c + 1 < vis_hi) ? p1 : 0.f;
            }
            sum0 += p0;
            sum1 += p1;
            const uint32_t hi = pack2(p0, p1, BF16);
            pk[(c - c0) >> 1] = hi;
            if constexpr (kSplitP)
              pk_lo[(c - c0) >> 1] =
                  pack2(p0 - low_as_float(hi, BF16), p1 - high_as_float(hi, BF16), BF16);
          }
          tmem_st_x16(tS + (c0 >> 1), pk);
          if constexpr (kSplitP) tmem_st_x16(tS + 64 + (c0 >> 1), pk_lo);
        }
        l = l * alpha + (sum0 + sum1);
        // O rescale (the previous P·V of this tile is complete: S_t(j) was issued
        // after it and s_full tracks all earlier MMAs).
        if (__any_sync(0xffffffffu, rescale && j != span.lo)) {
          const float a = (rescale && j != span.lo) ? alpha : 1.f;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t orow[32];
            tmem_ld_x32(tO + c0, orow);
#pragma unroll
            for (int c = 0; c < 32; ++c) orow[c] = __float_as_uint(__uint_as_float(orow[c]) * a);
            tmem_st_x32(tO + c0, orow);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_p_full(t));
      }
      if (!ok) break;
      // ---- epilogue: O / l and LSE for this tile
      ok = mbar_wait_warp(bar_o_full(t), o_cnt & 1u, wc, kSiteSmxOFull);
      ++o_cnt;
      if (!ok) break;
      tc_fence_after();
      const bool live = row < p.L;
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const size_t o_row = ((static_cast<size_t>(u.b) * p.L + row) * p.Hq + u.h) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t orow[32];
        tmem_ld_x32(tO + c0, orow);
        if (live) {
          if constexpr (OUT_F32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + o_row + c0);
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              dst[c >> 2] = make_float4(__uint_as_float(orow[c]) * inv_l,
                                        __uint_as_float(orow[c + 1]) * inv_l,
                                        __uint_as_float(orow[c + 2]) * inv_l,
                                        __uint_as_float(orow[c + 3]) * inv_l);
          } else {
            uint4* dst =
                reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + o_row + c0);
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
              uint4 w;
              w.x = pack2(__uint_as_float(orow[c]) * inv_l, __uint_as_float(orow[c + 1]) * inv_l, BF16);
              w.y = pack2(__uint_as_float(orow[c + 2]) * inv_l, __uint_as_float(orow[c + 3]) * inv_l, BF16);
              w.z = pack2(__uint_as_float(orow[c + 4]) * inv_l, __uint_as_float(orow[c + 5]) * inv_l, BF16);
              w.w = pack2(__uint_as_float(orow[c + 6]) * inv_l, __uint_as_float(orow[c + 7]) * inv_l, BF16);
              dst[c >> 3] = w;
            }
          }
        }
      }
      if (live && p.lse != nullptr) {
        const float lse = (l > 0.f) ? (m_ref + lg2_approx(l)) * 0.69314718055994531f : -INFINITY;
        p.lse[(static_cast<size_t>(u.b) * p.Hq + u.h) * p.L + row] = lse;
      }
      tc_fence_before();
      mbar_arrive(bar_o_free(t));
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

}  // namespace ex19
