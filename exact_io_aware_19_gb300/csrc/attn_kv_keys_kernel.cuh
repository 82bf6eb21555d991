// attn_kv_keys_kernel.cuh — the decode-shaped forward with the keys of a block on the
// TMEM lanes, for work items of at most 32 query rows (a few new tokens, times the
// query heads that share one K/V head).
//
// It computes what attn_kv_sm103_kernel computes for the same item (the last Lq
// positions of an Lk-long sequence, the same masks, key splits and partial outputs),
// the generation step that "What is memory-efficient attention for long context on
// 8x H100?" (section 1) names as bound by reading the whole KV cache. With only a few
// rows the row-per-lane layout leaves one thread to walk 128 scores per block while
// the rest of the warp idles; here the products are transposed so that each thread
// owns one key:
//   * S^T = K_j · Q^T: M = 128 keys (TMEM lanes), N = 16 or 32 query rows (columns).
//     A = the K slot (K-major), B = the Q tile (K-major, 32 rows).
//   * O^T += V_j^T · P^T: M = 128 (the d dimension; at d = 64 the second half of M
//     reads unrelated shared memory and those accumulator lanes are never read),
//     N = the query rows. A = the V slot read MN-major (the same layout the TMA
//     writes), B = P^T written by the softmax threads into shared memory in the
//     K-major 128-byte-swizzled layout. bf16 P is split into hi + lo operands (two
//     products) as in the other kernels; fp16 P is not.
//   * warps 0-3 (softmax, thread t = key t of the block): one score per query row per
//     block. All rows share one reference max per row (the weights of one product
//     must): a block whose scores exceed it by more than 2^8 is detected by a vote of
//     the four warps (a named barrier per block) and takes a slow path that reduces
//     the block maximum over all keys, moves the reference and rescales O^T and the
//     per-thread sums l. The sums are per thread and meet once, in the epilogue.
//   * warp 4 (producer): kv_produce, the ring of K/V slots of the one-tile kernel.
//   * warp 5 (MMA): O^T += V^T P^T(j) once P(j) is in shared memory, then S^T(j+2)
//     (two S buffers, two P buffers). Two orderings need no barrier of their own:
//     S^T(j+2) overwrites S^T(j) only after P·V(j) waited for P(j), which every
//     warp writes after reading S^T(j); and the commit of S^T(j) (s_full) tracks
//     P·V(j-2), issued before it, so a warp that has S^T(j) may overwrite P(j-2).
//   * Every wait is bounded; the four softmax warps leave the block loop together
//     (an abort bit rides on the per-block vote), so the named barriers never wait
//     for a warp that has left.
//   * Key splits (splits > 1) of items of at most 8 rows are combined by their
//     log-sum-exp inside this kernel, by whichever CTA of a work item stores its
//     partial result last; no CTA waits for another (32-row items leave their
//     partial results to the merge kernel). Each item has a 64-bit ticket in the workspace holding the call's
//     tag (bits 9 and up, a new value per call) and a count (bits 0-8). At its start
//     a CTA claims the ticket for this call (a compare-and-swap that replaces a word
//     with another tag, whatever an earlier call or a fresh workspace left there, by
//     tag << 9); after storing its partial O and LSE (and a fence) it adds 1. The CTA
//     whose add returns splits - 1 reads every split's partial result back from L2,
//     writes the item's O and LSE, and resets the count to 0 (so a graph replay with
//     the same tag starts from a claimed, empty ticket). Every CTA adds exactly once,
//     on error paths too.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <type_traits>

#include "attn_kv_kernel.cuh"

namespace ex19 {
namespace kv {

constexpr int kKeysRowsMax = 32;  // query rows per work item
constexpr int kKeysThreads = 192;  // 4 softmax warps + producer + MMA
constexpr int kKeysProducerWarp = 4;
constexpr int kKeysMmaWarp = 5;
constexpr uint32_t kKeysTmemCols = 128;  // S^T buffers [0, 32) and [32, 64), O^T [64, 96)
constexpr int kKeysPrefetchBlocks = 4;    // key blocks brought into L2 before the grid wait

enum : uint32_t {
  kSiteKeysMmaKFull = 0xA0001, kSiteKeysMmaVFull = 0xA0002, kSiteKeysMmaPFull = 0xA0003,
  kSiteKeysMmaQFull = 0xA0005, kSiteKeysMmaDrain = 0xA0006,
  kSiteKeysSmxSFull = 0xB0001, kSiteKeysSmxPvDone = 0xB0003, kSiteKeysSmxOFull = 0xB0004,
  kSiteKeysTicket = 0xB0005,
};

template <int D>
struct KeysGeometry {
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kBM * D * 2;             // 128 keys of K or V
  static constexpr int kChunkBytes = kBM * 128;              // 64 columns of such a tile
  static constexpr int kRowChunkBytes = kKeysRowsMax * 128;  // 64 columns of 32 rows
  static constexpr int kPBytes = 2 * kRowChunkBytes;         // P^T of one block: 128 keys x 32 rows
  // One CTA per SM with a deep ring: at d = 64, 8 slots (4 blocks in flight) measured
  // 29.3 against 30.3 us per 128k-key decode call for two CTAs per SM of 4 slots each.
  static constexpr int kSlots = (D == 64) ? 8 : 5;
  static constexpr int kCtasPerSm = 1;
  // The ring first, then P: at d = 64 the O^T product's second M half reads the 16 KiB
  // after a V slot, which for the last slot is the P region.
  static constexpr int kOffKV = 0;
  static constexpr int kOffP = kOffKV + kSlots * kTileBytes;  // [buffer 2][part 2 (hi, lo)]
  static constexpr int kOffQ = kOffP + 4 * kPBytes;
  static constexpr int kOffBar = kOffQ + kChunks * kRowChunkBytes;
  // full[S], empty[S], q_full, s_full[2], p_full[2], pv_done[2], o_full, drain
  static constexpr int kNumBars = 2 * kSlots + 9;
  // tmem base, abort flag, votes [2][4] bytes, the last-CTA flag of the merge
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffRed = kOffMisc + 32;            // [2][4 warps][32 rows] block maxima
  static constexpr int kOffLsum = kOffRed + 2 * 4 * kKeysRowsMax * 4;  // [4 warps][32 rows] sums
  static constexpr int kSmemUsed = kOffLsum + 4 * kKeysRowsMax * 4;
  static constexpr int kSmemBytes = kSmemUsed + 1024;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// The merge of a work item's key splits by the last of its CTAs (the 128 softmax
// threads; every split's partial result is in L2). Row r of the item:
// O = sum_s w_s O_s and LSE = m + log2(L) (base 2, stored as ln), with
// w_s = 2^(lse_s - m) / L, L = sum_s 2^(lse_s - m), m = max_s lse_s ("What is
// memory-efficient attention for long context on 8x H100?", section 4: attention in
// parts, combined by the log-sum-exp). An empty split (lse = -inf, O = 0) has weight
// 0; a row with no visible key gets O = 0 and LSE = -inf.
// The item's output is cut into 16-byte quads (rows x D/4). With at most 128 quads,
// `slots` = 128 / quads threads share a quad and take every slots-th split; each
// thread loads up to kPer of its splits' LSEs and O quads at once (a reload from L2
// costs about a microsecond, so a merge of a call's splits is one or two round
// trips), folds them in with a running maximum, and the slots of a quad meet in
// shared memory in slot order (the result does not depend on which CTA merges). With more quads each thread takes quads
// t, t + 128, ... alone. `scratch` holds 6 floats per (slot, quad).
template <int D, bool BF16, int kPer>
__device__ __forceinline__ void keys_merge_splits(const KvParams& p, const KvItem& it, int rows,
                                                  int t, float* scratch, int out_f32) {
  constexpr int kQuads = D / 4;
  const size_t nrows = static_cast<size_t>(p.B) * p.Hq * p.Lq;
  const int S = p.splits;
  const int nq = rows * kQuads;
  const int slots = (nq < 128) ? 128 / nq : 1;
  for (int base = 0; base < nq; base += 128 / slots) {
    const int qd = base + t % (128 / slots), slot = t / (128 / slots);
    const bool live = qd < nq && slot < slots;
    const int r = qd / kQuads, c4 = qd % kQuads;
    const int qi = it.i0 + r / p.group;
    const int h = it.g * p.group + r % p.group;
    const size_t row = (static_cast<size_t>(it.b) * p.Hq + h) * p.Lq + qi;
    float m = -INFINITY, l = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = slot; live && s0 < S; s0 += slots * kPer) {
      float ls[kPer];
      float4 ov[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int sp = s0 + u * slots;
        ls[u] = -INFINITY;
        ov[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (sp < S) {
          ls[u] = __ldcg(p.lse_part + static_cast<size_t>(sp) * nrows + row);
          ov[u] = __ldcg(reinterpret_cast<const float4*>(p.o_part + (static_cast<size_t>(sp) * nrows + row) * D) + c4);
        }
      }
      float mc = m;
#pragma unroll
      for (int u = 0; u < kPer; ++u) mc = fmaxf(mc, ls[u]);
      if (mc != -INFINITY) {
        const float f = exp2f(m - mc);  // 0 while m is -inf
        l *= f;
        a = make_float4(a.x * f, a.y * f, a.z * f, a.w * f);
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const float w = exp2f(ls[u] - mc);  // 0 for an empty split
          l += w;
          a = make_float4(fmaf(w, ov[u].x, a.x), fmaf(w, ov[u].y, a.y), fmaf(w, ov[u].z, a.z),
                          fmaf(w, ov[u].w, a.w));
        }
        m = mc;
      }
    }
    if (slots > 1) {  // uniform: the slots of a quad meet in shared memory
      float* mine = scratch + 6 * (slot * nq + qd);
      if (live && slot > 0) {
        mine[0] = m;
        mine[1] = l;
        mine[2] = a.x;
        mine[3] = a.y;
        mine[4] = a.z;
        mine[5] = a.w;
      }
      named_barrier(1, 128);
      if (live && slot == 0) {
        for (int o = 1; o < slots; ++o) {
          const float* q = scratch + 6 * (o * nq + qd);
          const float mm = fmaxf(m, q[0]);
          if (mm != -INFINITY) {
            const float f1 = exp2f(m - mm), f2 = exp2f(q[0] - mm);
            l = l * f1 + q[1] * f2;
            a = make_float4(a.x * f1 + q[2] * f2, a.y * f1 + q[3] * f2, a.z * f1 + q[4] * f2,
                            a.w * f1 + q[5] * f2);
            m = mm;
          }
        }
      }
    }
    if (live && slot == 0) {
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      const float o4[4] = {a.x * inv, a.y * inv, a.z * inv, a.w * inv};
      const size_t oi = ((static_cast<size_t>(it.b) * p.Lq + qi) * p.Hq + h) * D + 4 * c4;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (out_f32)
          static_cast<float*>(p.o)[oi + j] = o4[j];
        else if constexpr (BF16)
          static_cast<__nv_bfloat16*>(p.o)[oi + j] = __float2bfloat16_rn(o4[j]);
        else
          static_cast<__half*>(p.o)[oi + j] = __float2half_rn(o4[j]);
      }
      if (c4 == 0 && p.lse != nullptr)
        p.lse[row] = (l > 0.f) ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  }
}

// NQ: the query rows a work item may have (1, 8 or 32; the products use N = max(NQ, 16)).
template <int D, bool BF16, bool PAGED, int NQ>
__global__ void __launch_bounds__(kKeysThreads, KeysGeometry<D>::kCtasPerSm)
    attn_kv_keys_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const KvParams p, int out_f32) {
  static_assert(NQ == 1 || NQ == 8 || NQ == 32, "rows per item");
  using G = KeysGeometry<D>;
  constexpr int S = G::kSlots;
  constexpr int kN = NQ < 16 ? 16 : NQ;  // N of both products
  constexpr bool kSplitP = BF16;         // bf16 P as hi + lo operands
  constexpr float kThresh = 8.0f;        // log2 units of max growth before a rescale
  constexpr bool kSelfMerge = NQ <= 8;   // key splits merged by the item's last CTA

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sKV = sbase + G::kOffKV;
  const uint32_t sP = sbase + G::kOffP;
  const uint32_t sQ = sbase + G::kOffQ;
  const uint32_t bars = sbase + G::kOffBar;
  auto bar_full = [&](uint32_t s) { return bars + 8u * s; };
  auto bar_empty = [&](uint32_t s) { return bars + 8u * (S + s); };
  const uint32_t bar_q_full = bars + 8u * (2 * S);
  auto bar_s_full = [&](uint32_t b) { return bars + 8u * (2 * S + 1 + b); };
  auto bar_p_full = [&](uint32_t b) { return bars + 8u * (2 * S + 3 + b); };
  auto bar_pv_done = [&](uint32_t b) { return bars + 8u * (2 * S + 5 + b); };
  const uint32_t bar_o_full = bars + 8u * (2 * S + 7);
  const uint32_t bar_drain = bars + 8u * (2 * S + 8);
  auto p_buf = [&](uint32_t b, int part) { return sP + (2u * b + part) * G::kPBytes; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + G::kOffMisc + 4);
  volatile uint8_t* votes = smem + G::kOffMisc + 8;  // [2 buffers][4 warps]
  float* red = reinterpret_cast<float*>(smem + G::kOffRed);
  float* lsum = reinterpret_cast<float*>(smem + G::kOffLsum);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_q_full, 1);
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(bar_s_full(b), 1);
      mbar_init(bar_p_full(b), 128);
      mbar_init(bar_pv_done(b), 1);
    }
    mbar_init(bar_o_full, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kKeysProducerWarp && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    // The first blocks of this CTA's keys, into L2 while the kernel before this one
    // ends (each CTA of the previous decode call lets this grid start once its block
    // loop is done).
    if constexpr (!PAGED) kv_prefetch_first_blocks<D>(p, &tm_k, &tm_v, kKeysPrefetchBlocks);
  }
  // A programmatic dependent launch: the previous kernel's writes are visible past
  // this point; TMEM is allocated only after it (as in the one-tile kernel).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (warp == kKeysMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kKeysTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const KvItem it = kv_item<PAGED>(p);
  const int nblocks = max(0, it.hi - it.lo);
  volatile uint32_t* merge_flag = reinterpret_cast<volatile uint32_t*>(smem + G::kOffMisc + 16);
  // items of at most 8 rows merge their splits here; 32-row items leave it to the
  // merge kernel launched after this one
  unsigned long long* ticket =
      (kSelfMerge && p.splits > 1) ? p.tickets + blockIdx.x / p.splits : nullptr;
  if (ticket != nullptr && threadIdx.x == 0) {
    // claim the item's ticket for this call (the same thread adds to it at the end)
    const unsigned long long w = __ldcg(ticket);
    if ((w & ~511ull) != p.ticket_base) atomicCAS(ticket, w, p.ticket_base);
  }

  WaitCtl wc;
  wc.abort_flag = abort_flag;
  wc.status = p.status;
  wc.set_limit(p.wait_limit_ns);
  wc.unit = blockIdx.x;
  if (it.bad && threadIdx.x == 0) record_error(wc, kStatusInvalidArg, kSiteBadSeqLen);

  if (warp == kKeysProducerWarp) {
    kv_produce<PAGED, D>(p, it, nblocks, &tm_q, &tm_k, &tm_v, sQ, G::kRowChunkBytes, sKV, S, bars,
                         wc, lane);
  } else if (warp == kKeysMmaWarp) {
    // ------------------------------------------------------------- MMA issuer
    if (nblocks > 0) {
      constexpr uint32_t idesc_s = idesc_f16_f32acc_ab(BF16, kBM, kN, false, false);
      constexpr uint32_t idesc_o = idesc_f16_f32acc_ab(BF16, kBM, kN, true, false);
      const uint64_t dk = sdesc_sw128(sKV, 16, 1024);               // K slots as A, K-major
      const uint64_t dq = sdesc_sw128(sQ, 16, 1024);                // Q rows as B, K-major
      const uint64_t dv = sdesc_sw128(sKV, G::kChunkBytes, 1024);   // V slots as A, MN-major
      const uint32_t mO = tmem_base + 64;
      auto slot_of = [&](uint32_t idx) { return idx % S; };
      auto par_of = [&](uint32_t idx) { return (idx / S) & 1u; };
      // S^T(jj) = K_j · Q^T into buffer jj & 1 (S^T(jj - 2) has been read: see the
      // header).
      auto issue_s = [&](int jj) __attribute__((always_inline)) -> bool {
        const uint32_t kidx = 2u * jj, b = jj & 1;
        if (!mbar_wait_warp(bar_full(slot_of(kidx)), par_of(kidx), wc, kSiteKeysMmaKFull)) return false;
        tc_fence_after();
        const uint32_t mS = tmem_base + 32u * b;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ka = (kk >> 2) * G::kChunkBytes + (kk & 3) * 32;
          const uint32_t kb = (kk >> 2) * G::kRowChunkBytes + (kk & 3) * 32;
          mma_ss_elect(mS, dk + ((slot_of(kidx) * G::kTileBytes + ka) >> 4), dq + (kb >> 4), idesc_s,
                       kk > 0 ? 1u : 0u);
        }
        mma_commit_elect(bar_s_full(b));
        mma_commit_elect(bar_empty(slot_of(kidx)));
        return true;
      };
      // O^T += V_j^T · P^T(jj) once P(jj) is in buffer jj & 1; releases V_j.
      auto issue_pv = [&](int jj) __attribute__((always_inline)) -> bool {
        const uint32_t vidx = 2u * jj + 1u, b = jj & 1;
        if (!mbar_wait_warp(bar_full(slot_of(vidx)), par_of(vidx), wc, kSiteKeysMmaVFull)) return false;
        if constexpr (PAGED) {
          // Rows past the sequence in its last block: the part of a partial page the
          // TMA did load holds arbitrary cache contents; make every such V row 0.
          const int r0 = it.Lk - (it.lo + jj) * kBN;
          if (r0 < kBN) {
            const uint32_t base = sKV + slot_of(vidx) * G::kTileBytes;
            for (int idx = lane; idx < (kBN - r0) * 8 * G::kChunks; idx += 32) {
              const int c = idx / ((kBN - r0) * 8), rem = idx % ((kBN - r0) * 8);
              st_shared_zero16(base + c * G::kChunkBytes + (r0 + rem / 8) * 128 + (rem % 8) * 16);
            }
            fence_proxy_async_shared();
            __syncwarp();
          }
        }
        if (!mbar_wait_warp(bar_p_full(b), (jj >> 1) & 1u, wc, kSiteKeysMmaPFull)) return false;
        tc_fence_after();
        const uint64_t dvs = dv + ((slot_of(vidx) * G::kTileBytes) >> 4);
#pragma unroll
        for (int part = 0; part < (kSplitP ? 2 : 1); ++part) {
          const uint64_t dp = sdesc_sw128(p_buf(b, part), 16, 1024);  // P^T rows as B, K-major
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint32_t kb = (kk >> 2) * G::kRowChunkBytes + (kk & 3) * 32;
            mma_ss_elect(mO, dvs + ((kk * 2048) >> 4), dp + (kb >> 4), idesc_o,
                         (jj == 0 && part == 0 && kk == 0) ? 0u : 1u);
          }
        }
        mma_commit_elect(bar_pv_done(b));
        mma_commit_elect(bar_empty(slot_of(vidx)));
        return true;
      };
      bool ok = mbar_wait_warp(bar_q_full, 0, wc, kSiteKeysMmaQFull);
      if (ok) {
        tc_fence_after();
        ok = issue_s(0);
        if (ok && nblocks > 1) ok = issue_s(1);
        for (int jj = 0; ok && jj < nblocks; ++jj) {
          ok = issue_pv(jj);
          if (ok && jj + 2 < nblocks) ok = issue_s(jj + 2);
        }
        if (ok) mma_commit_elect(bar_o_full);
      }
    }
    mma_commit_elect(bar_drain);
    mbar_wait_drain(bar_drain, 0, wc, kSiteKeysMmaDrain);
  } else {
    // -------------------------------------------------------- softmax warps
    const int t = threadIdx.x;  // key of the block, TMEM lane (and the d row of O^T)
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int rows = it.bad ? 0 : (it.i1 - it.i0) * p.group;  // valid query rows (<= NQ)
    const int Lk = it.Lk;
    const int off = Lk - p.Lq;
    const int wr = right_bound(p);
    const float C = p.score_log2;
    const float Cs = (p.negate_scores != 0) ? -C : C;
    float mref[NQ], l[NQ];
#pragma unroll
    for (int c = 0; c < NQ; ++c) {
      mref[c] = -INFINITY;
      l[c] = 0.f;
    }
    // the key-of-thread byte offset in a P^T operand (chunk of 64 keys, swizzled
    // 16-byte granule of the row); the row part is added per row
    const uint32_t p_key = static_cast<uint32_t>((t >> 6) * G::kRowChunkBytes + (t & 7) * 2);
    const uint32_t p_gran = static_cast<uint32_t>((t & 63) >> 3);
    bool ok = true;
    // Blocks [ja, jb) cross no mask boundary (as in the one-tile kernel).
    int ja = 0, jb = nblocks;
    {
      const int pos_min = off + it.i0, pos_max = off + it.i1 - 1;
      if (p.window_left >= 0) {
        const int first = pos_max - p.window_left;
        if (first > 0) ja = max(ja, (first + kBN - 1) / kBN - it.lo);
      }
      jb = min(jb, Lk / kBN - it.lo);
      if (wr >= 0) {
        const int last = pos_min + wr - (kBN - 1);
        jb = min(jb, last >= 0 ? last / kBN + 1 - it.lo : 0);
      }
      ja = min(max(ja, 0), nblocks);
      jb = max(jb, ja);
    }
    for (int jj = 0; jj < nblocks; ++jj) {
      const uint32_t b = jj & 1;
      float x[NQ];
      bool exceed = false;
      if (ok) {
        ok = mbar_wait_warp(bar_s_full(b), (jj >> 1) & 1u, wc, kSiteKeysSmxSFull);
        if (ok) {
          tc_fence_after();
          uint32_t sr[NQ];
          tmem_ld_n<NQ>(tmem_base + lane_off + 32u * b, sr);
          const bool masked = jj < ja || jj >= jb;
          const int key = (it.lo + jj) * kBN + t;
#pragma unroll
          for (int c = 0; c < NQ; ++c) {
            x[c] = __uint_as_float(sr[c]) * Cs;
            bool vis = c < rows;
            if (masked) {
              const int pos = off + it.i0 + c / p.group;
              vis = vis && key < Lk && (wr < 0 || key <= pos + wr) &&
                    (p.window_left < 0 || key >= pos - p.window_left);
            }
            if (!vis) x[c] = -INFINITY;
            exceed = exceed || x[c] > mref[c] + kThresh;
          }
        }
      }
      // the vote: bit 0 a score above the reference, bit 1 this warp stopped
      const bool any = __any_sync(0xffffffffu, exceed);
      if (lane == 0) votes[b * 4 + warp] = static_cast<uint8_t>((any ? 1u : 0u) | ((ok && !*abort_flag) ? 0u : 2u));
      named_barrier(1, 128);
      const uint32_t v4 = *reinterpret_cast<volatile uint32_t*>(votes + b * 4);
      if (v4 & 0x02020202u) {
        ok = false;
        break;
      }
      if (v4 & 0x01010101u) {
        // slow path: the block maximum of every row over all 128 keys
        float* rb = red + b * 4 * kKeysRowsMax;
#pragma unroll
        for (int c = 0; c < NQ; ++c) {
          const float m = warp_max(x[c]);
          if (lane == 0) rb[warp * kKeysRowsMax + c] = m;
        }
        named_barrier(1, 128);
        float alpha[NQ];
        bool resc = false;
#pragma unroll
        for (int c = 0; c < NQ; ++c) {
          const float bm = fmaxf(fmaxf(rb[c], rb[kKeysRowsMax + c]),
                                 fmaxf(rb[2 * kKeysRowsMax + c], rb[3 * kKeysRowsMax + c]));
          alpha[c] = 1.f;
          if (bm > mref[c] + kThresh) {
            alpha[c] = ex2_approx(mref[c] - bm);  // 0 when mref is -inf
            mref[c] = bm;
            resc = true;
          }
          l[c] *= alpha[c];
        }
        if (resc && jj > 0) {  // O^T lanes = d rows, columns = query rows
          ok = mbar_wait_warp(bar_pv_done((jj - 1) & 1), ((jj - 1) >> 1) & 1u, wc, kSiteKeysSmxPvDone);
          if (ok) {
            tc_fence_after();
            uint32_t orow[NQ];
            tmem_ld_n<NQ>(tmem_base + lane_off + 64u, orow);
#pragma unroll
            for (int c = 0; c < NQ; ++c) orow[c] = __float_as_uint(__uint_as_float(orow[c]) * alpha[c]);
            tmem_st_n<NQ>(tmem_base + lane_off + 64u, orow);
            tmem_st_wait();
          }
        }
      }
      if (!ok) continue;  // the next vote carries the stop
      // P = 2^(x - m) for this key and every row; l per thread
#pragma unroll
      for (int c = 0; c < NQ; ++c) {
        const float mu = (mref[c] == -INFINITY) ? 0.f : mref[c];
        const float pv = ex2_approx(x[c] - mu);  // 0 for masked keys (x = -inf)
        l[c] += pv;
        if (c < rows) {
          const uint32_t a = p_key + c * 128 + ((p_gran ^ (c & 7)) << 4);
          if constexpr (kSplitP) {
            const __nv_bfloat16 hi = __float2bfloat16_rn(pv);
            const __nv_bfloat16 lo = __float2bfloat16_rn(pv - __bfloat162float(hi));
            st_shared_u16(p_buf(b, 0) + a, __bfloat16_as_ushort(hi));
            st_shared_u16(p_buf(b, 1) + a, __bfloat16_as_ushort(lo));
          } else {
            st_shared_u16(p_buf(b, 0) + a, __half_as_ushort(__float2half_rn(pv)));
          }
        }
      }
      fence_proxy_async_shared();
      tc_fence_before();
      mbar_arrive(bar_p_full(b));
    }
    // ---- epilogue: the row sums over the 128 key threads, then O / l and the LSE
#pragma unroll
    for (int c = 0; c < NQ; ++c) {
      const float s = warp_sum(l[c]);
      if (lane == 0) lsum[warp * kKeysRowsMax + c] = s;
    }
    if (ok && nblocks > 0) {
      ok = mbar_wait_warp(bar_o_full, 0, wc, kSiteKeysSmxOFull);
      if (ok) tc_fence_after();
    }
    // This CTA has read all of its keys: the next kernel on the stream may start (its
    // CTAs still wait for this grid's end before touching global memory or TMEM).
    // Not when a merge kernel follows (it measured slower launched early).
    if constexpr (kSelfMerge) asm volatile("griddepcontrol.launch_dependents;");
    named_barrier(1, 128);
    if (ok) {
      float lt[NQ];
#pragma unroll
      for (int c = 0; c < NQ; ++c)
        lt[c] = (lsum[c] + lsum[kKeysRowsMax + c]) + (lsum[2 * kKeysRowsMax + c] + lsum[3 * kKeysRowsMax + c]);
      uint32_t orow[NQ];
      if (nblocks > 0) {
        tmem_ld_n<NQ>(tmem_base + lane_off + 64u, orow);
      } else {
#pragma unroll
        for (int c = 0; c < NQ; ++c) orow[c] = 0u;
      }
      const bool partial = p.splits > 1;
      const size_t nrows = static_cast<size_t>(p.B) * p.Hq * p.Lq;
#pragma unroll
      for (int c = 0; c < NQ; ++c) {
        if (c >= rows) continue;
        const int qi = it.i0 + c / p.group;
        const int h = it.g * p.group + c % p.group;
        const size_t row = (static_cast<size_t>(it.b) * p.Hq + h) * p.Lq + qi;  // LSE index
        const float inv_l = (lt[c] > 0.f) ? 1.f / lt[c] : 0.f;
        if (t < D) {
          const float o = __uint_as_float(orow[c]) * inv_l;
          if (partial) {
            p.o_part[(static_cast<size_t>(it.split) * nrows + row) * D + t] = o;
          } else {
            const size_t oi = ((static_cast<size_t>(it.b) * p.Lq + qi) * p.Hq + h) * D + t;
            if (out_f32)
              static_cast<float*>(p.o)[oi] = o;
            else if constexpr (BF16)
              static_cast<__nv_bfloat16*>(p.o)[oi] = __float2bfloat16_rn(o);
            else
              static_cast<__half*>(p.o)[oi] = __float2half_rn(o);
          }
        }
        if (t == c) {
          const float lse2 = (lt[c] > 0.f) ? mref[c] + lg2_approx(lt[c]) : -INFINITY;  // base 2
          if (partial)
            p.lse_part[static_cast<size_t>(it.split) * nrows + row] = lse2;
          else if (p.lse != nullptr)
            p.lse[row] = (lt[c] > 0.f) ? lse2 * 0.69314718055994531f : -INFINITY;
        }
      }
    }
    if (ticket != nullptr) {
      // ---- the split merge: this CTA's partial result is stored; take a ticket
      __threadfence();  // each thread's partial stores, before the add below
      named_barrier(1, 128);
      if (t == 0) {
        const unsigned long long prev = atomicAdd(ticket, 1ull);
        const unsigned long long n = prev & 511ull;  // CTAs of the item that added before
        uint32_t last = 0u;
        if ((prev & ~511ull) != p.ticket_base || n >= static_cast<unsigned long long>(p.splits)) {
          record_error(wc, kStatusWorkspace, kSiteKeysTicket);  // another call shares the workspace
        } else if (n + 1 == static_cast<unsigned long long>(p.splits)) {
          last = 1u;
          atomicExch(ticket, p.ticket_base);  // empty again, for a replay with this tag
        }
        *merge_flag = last;
      }
      named_barrier(1, 128);
      if (*merge_flag != 0u) {  // uniform over the 128 threads (the merge has barriers)
        __threadfence();  // the other CTAs' partial results, after their adds
        // kPer: splits of one thread in flight at once. A one-row item shares each
        // column quad among 128 / (D / 4) threads (8 at d = 64: 64 splits in one round
        // trip with 8 each), and the smaller body is fetched faster (the merge code
        // runs cold: once per call, on one CTA).
        keys_merge_splits<D, BF16, (NQ == 1 ? 8 : 24)>(p, it, rows, t, reinterpret_cast<float*>(smem + G::kOffKV), out_f32);
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kKeysMmaWarp) {
    __syncwarp();
    tmem_dealloc(tmem_base, kKeysTmemCols);
  }
}

}  // namespace kv
}  // namespace ex19
