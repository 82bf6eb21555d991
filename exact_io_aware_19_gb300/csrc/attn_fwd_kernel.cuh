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
//   * warps 9, 10 (MMA, tile 0 / tile 1): each warp runs its issue loop
//              warp-uniformly and one lane, picked by elect.sync, issues each
//              tcgen05.mma. S_t = Q_t K_jᵀ goes to TMEM (fp32, 128 columns per
//              tile); O_t += P_t V_j reads P_t from TMEM (16-bit; in columns of its
//              own at d = 64 fp16, aliased over S_t otherwise) and V_j from shared
//              memory. One issuer per tile, so one tile's softmax overlaps the
//              other tile's MMAs and neither tile's MMAs queue behind the other's.
//   * warps 0-3 / 4-7 (softmax, tile 0 / tile 1): one thread per query row (TMEM
//              lane). Loads its row of S, masks boundary blocks, keeps the running
//              max m (base-2 units) and sum l, writes P = 2^(x - m) back to TMEM,
//              rescales its O row when m grows by more than a threshold (2^1 with
//              packed fp16 exponentials, 2^8 otherwise), and at the end of the unit
//              writes O / l and LSE.
//   * Alternating mode (ALT, for small problems whose time is the longest row
//     tile's chain of key blocks): a work unit is one 128-row tile, and both
//     pipelines (MMA warp, softmax warps, TMEM columns) work on it, pipeline t
//     taking the key blocks lo + t, lo + t + 2, ... with its own running max, sum
//     and O. At the end tile 1's softmax warps hand their max and sum to tile 0's
//     through shared memory, and tile 0's warps read O_1 from TMEM and write the
//     combination (the merge of attention computed in parts: with m = max(m_0,
//     m_1), O = (2^(m_0 - m) O_0 + 2^(m_1 - m) O_1) / (2^(m_0 - m) l_0 +
//     2^(m_1 - m) l_1)). A tile's chain is half as long.
//   * Dynamic scheduling (when the call gives a counter, p.sched): the producer
//     takes the next unit rank from a global atomic counter when it starts a unit
//     and passes it to the MMA and softmax warps through a 4-entry queue in shared
//     memory. Ranks stay heaviest first; a CTA on a faster SM simply takes more
//     units, so the grid ends within about one small unit of the mean (a static deal
//     left CTAs finishing from 7.9 to 8.6 ms on one causal L = 131072 call, the same
//     units running up to 18 % slower on some SMs).
//   * Launch order: a programmatic dependent launch. The prologue touches shared
//     memory only (with the static deal the producer also asks for its first
//     unit's tiles in L2, a hint), then griddepcontrol.wait precedes the TMEM
//     allocation and every global access; once the producer has issued its last
//     load, the CTA lets the next kernel on the stream start.
//   * Every wait is bounded (globaltimer); a wait that runs out records a timeout
//     in the status word and every role leaves its loop, so the CTA still frees
//     its TMEM and exits.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <type_traits>

#include "attn_params.h"
#include "row_ops.cuh"
#include "sm103_ptx.cuh"
#include "tmem_io.cuh"
#include "vscale.cuh"

namespace ex19 {

constexpr int kBM = 128;             // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;             // keys per K/V block
constexpr int kTilesPerUnit = 2;     // query tiles per work unit
constexpr int kUnitRows = kBM * kTilesPerUnit;
constexpr int kThreads = 352;        // 8 softmax warps + producer warp + 2 MMA warps
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;          // warps 9 and 10: MMA issuers of tile 0 and tile 1
constexpr uint32_t kTmemCols = 512;  // S0 [0,128) S1 [128,256) O0 [256,..) O1 [384,..)
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when m grows > 2^8

// Wait sites (for the status word): role << 16 | site
enum : uint32_t {
  kSiteProdEmpty = 0x10001, kSiteProdQFree = 0x10002,
  kSiteMmaQFull = 0x20001, kSiteMmaKFull = 0x20002, kSiteMmaVFull = 0x20003,
  kSiteMmaPFull = 0x20004, kSiteMmaOFree = 0x20005, kSiteMmaDrain = 0x20006,
  kSiteMmaSFree = 0x20007,
  kSiteSmxSFull = 0x30001, kSiteSmxOFull = 0x30002, kSiteSmxPvDone = 0x30003,
  kSiteDrainLoads = 0x40001, kSiteUnitQueue = 0x40002,
};

constexpr int kUnitQueue = 4;  // dynamic scheduling: unit ranks in flight between the roles
constexpr int kPrefetchBlocks = 4;  // key blocks of the first unit brought into L2 before the grid wait
constexpr int kUnitReaders = 2 + 8;  // the MMA warps and the softmax warps read each entry

template <int D>
struct Geometry {
  static constexpr int kChunks = D / 64;          // 64-element (128-byte) swizzle boxes per row
  static constexpr int kChunkBytes = kBM * 128;   // 128 rows x 128 bytes
  static constexpr int kTileBytes = kBM * D * 2;  // one 128-row tile of Q, K or V
  static constexpr int kSlots = (D == 64) ? 8 : 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kTilesPerUnit * kTileBytes;
  static constexpr int kOffBar = kOffKV + kSlots * kTileBytes;
  // barriers: full[S], empty[S], q_full, q_free, s_full[2], p_full[2], o_full[2], o_free[2],
  // drain, s_free[2], pv_done[2], p_half[2], merge_ready, merge_free (ALT),
  // unit queue full[4], empty[4] (dynamic scheduling)
  static constexpr int kNumBars = 2 * kSlots + 19 + 2 * kUnitQueue;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kOffXchg = kOffMisc + 16;           // ALT: [128 rows] (max, sum) of tile 1
  static constexpr int kOffUq = kOffXchg + kBM * 8;        // unit queue: [4] unit ranks
  static constexpr int kSmemUsed = kOffUq + kUnitQueue * 4;
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
// heavy-first ranking (causal: the last row blocks see the most keys). ALT: a unit
// is one 128-row tile, given to both pipelines.
// The unit of rank r (rank 0 = the heaviest).
template <bool ALT>
__device__ __forceinline__ void unit_from_rank(const FwdParams& p, long long r, Unit& u) {
  const int BH = p.B * p.Hq;
  const int mb = p.units_per_bh - 1 - static_cast<int>(r / BH);
  const int bh = static_cast<int>(r % BH);
  u.b = bh / p.Hq;
  u.h = bh % p.Hq;
  u.g = u.h / (p.Hq / p.Hkv);
  u.lo = 0x7fffffff;
  u.hi = 0;
  for (int t = 0; t < kTilesPerUnit; ++t) {
    u.t[t] = tile_span(p, ALT ? mb * kBM : mb * kUnitRows + t * kBM);
    if (u.t[t].lo < u.t[t].hi) {
      u.lo = min(u.lo, u.t[t].lo);
      u.hi = max(u.hi, u.t[t].hi);
    }
  }
}

template <bool ALT>
__device__ __forceinline__ bool unit_of(const FwdParams& p, int k, Unit& u) {
  const int G = gridDim.x;
  const int c = blockIdx.x;
  const long long r = static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - c) : c);
  if (r >= p.num_units) return false;
  unit_from_rank<ALT>(p, r, u);
  return true;
}

__device__ __forceinline__ bool has_block(const TileSpan& s, int j) { return j >= s.lo && j < s.hi; }

// The key blocks [a, b) of a tile's span [lo, hi) that cross no mask boundary:
// every key visible to every row of the tile (no ragged tail, wholly below the
// causal diagonal, wholly inside the left window). Blocks [lo, a) and [b, hi) are
// the masked ones: the window's first blocks and the diagonal or tail block.
__device__ __forceinline__ void unmasked_blocks(const FwdParams& p, const TileSpan& s, int& a, int& b) {
  a = s.lo;
  if (p.window_left >= 0) {  // key0 >= row0 + kBM - 1 - window_left
    const int first = s.row0 + kBM - 1 - p.window_left;
    if (first > 0) a = max(a, (first + kBN - 1) / kBN);
  }
  b = min(s.hi, p.L / kBN);  // key0 + kBN <= L
  if (p.causal) b = min(b, (s.row0 >= kBN - 1) ? (s.row0 - (kBN - 1)) / kBN + 1 : 0);  // key0 + kBN - 1 <= row0
  a = min(a, s.hi);
  b = max(b, a);
}

// PV16 (bf16 inputs only): V is the call's fp16 copy scaled per (batch, K/V head)
// by 2^e (vscale.cuh), P is fp16 and P·V one fp16 product; the output is scaled back.
template <int D, bool BF16, bool OUT_F32, bool PV16 = false, bool ALT = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_sm103_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using G = Geometry<D>;
  constexpr int S = G::kSlots;
  static_assert(!PV16 || BF16, "the fp16 copy of V is for bfloat16 inputs");
  // bf16 P is split into hi + lo halves (two P·V MMAs) so that rounding P to 8
  // significant bits does not dominate the output error; fp16 P has 11 bits.
  constexpr bool kSplitP = BF16 && !PV16;
  // P in fp16: the P·V product's operands (P, V or its fp16 copy) are fp16.
  constexpr bool kP16 = !kSplitP;
  // Packed fp16 exponentials (fp16 inputs): x is rounded to fp16 before 2^x, so x
  // must stay small where P is large; the reference max is then moved whenever
  // the row max grows by more than 2^1 instead of 2^8. With the fp16 copy of V the
  // exponentials are fp32 (l summed from them, P rounded to fp16 for the product):
  // measured on one GB300 both faster at d = 128 (GQA 32/8 L = 131072 95.3 against
  // 98.3 ms) and exact in the LSE to ~1e-6 instead of ~7e-4.
  constexpr bool kF16Exp = !BF16;
  constexpr float kThresh = kF16Exp ? 1.0f : kRescaleThreshold;
  // TMEM columns. With P over S (d = 128, or bf16 whose split P needs 128 columns):
  // S_t = [128t, 128t+128), P_t aliased over S_t, O_t = [256+128t, ...). With a
  // separate P region (d = 64, fp16 P): S_t = [128t, ...), P_t = [256+64t, 256+64t+64),
  // O_t = [384+64t, 384+64t+64) — all 512 columns.
  constexpr bool kSeparateP = (D == 64) && kP16;
  // Separate P: the softmax releases the first 64 keys of P (p_half) before it
  // computes the rest, and the first four P·V MMAs run under that second half.
  constexpr bool kHalves = kSeparateP;
  constexpr uint32_t kColS0 = 0, kStrideS = 128;
  constexpr uint32_t kColP0 = kSeparateP ? 256 : 0, kStrideP = kSeparateP ? 64 : 128;
  constexpr uint32_t kColO0 = kSeparateP ? 384 : 256, kStrideO = kSeparateP ? 64 : 128;
  static_assert(!ALT || kSeparateP, "the alternating mode is built for the separate-P layout");

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
  auto bar_s_free = [&](int t) { return bars + 8u * (2 * S + 11 + t); };
  auto bar_pv_done = [&](int t) { return bars + 8u * (2 * S + 13 + t); };
  auto bar_p_half = [&](int t) { return bars + 8u * (2 * S + 15 + t); };
  const uint32_t bar_merge_ready = bars + 8u * (2 * S + 17);  // ALT: tile 1's max and sum are written
  const uint32_t bar_merge_free = bars + 8u * (2 * S + 18);   // ALT: tile 0 has read them and O_1
  float2* xchg = reinterpret_cast<float2*>(smem + G::kOffXchg);
  auto bar_uq_full = [&](int i) { return bars + 8u * (2 * S + 19 + i); };
  auto bar_uq_empty = [&](int i) { return bars + 8u * (2 * S + 19 + kUnitQueue + i); };
  volatile int* uq = reinterpret_cast<volatile int*>(smem + G::kOffUq);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + G::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), kTilesPerUnit);  // one release per tile
    }
    mbar_init(bar_q_full, 1);
    mbar_init(bar_q_free, kTilesPerUnit);
    for (int t = 0; t < kTilesPerUnit; ++t) {
      mbar_init(bar_s_full(t), 1);
      mbar_init(bar_p_full(t), kBM);
      mbar_init(bar_o_full(t), 1);
      mbar_init(bar_o_free(t), kBM);
    }
    mbar_init(bar_drain, kTilesPerUnit);
    for (int t = 0; t < kTilesPerUnit; ++t) {
      mbar_init(bar_s_free(t), kBM);
      mbar_init(bar_pv_done(t), 1);
      mbar_init(bar_p_half(t), kBM);
    }
    mbar_init(bar_merge_ready, kBM);
    mbar_init(bar_merge_free, kBM);
    for (int i = 0; i < kUnitQueue; ++i) {
      mbar_init(bar_uq_full(i), 1);
      mbar_init(bar_uq_empty(i), kUnitReaders);
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    Unit u0;
    if (p.sched == nullptr && unit_of<ALT>(p, 0, u0)) {
      // With the static deal the first unit is known here: its Q tiles and first key
      // blocks go to L2 while the kernel before this one ends (the previous call's
      // CTAs let this grid start once their loads are issued). A prefetch is only a
      // hint; the loads after griddepcontrol.wait read what that kernel left.
      for (int t = 0; t < kTilesPerUnit; ++t)
        if (u0.t[t].lo < u0.t[t].hi)
          for (int c = 0; c < G::kChunks; ++c) tma_prefetch_l2_4d(&tm_q, c * 64, u0.h, u0.t[t].row0, u0.b);
      for (int j = u0.lo; j < min(u0.hi, u0.lo + kPrefetchBlocks); ++j)
        for (int c = 0; c < G::kChunks; ++c) {
          tma_prefetch_l2_4d(&tm_k, c * 64, u0.g, j * kBN, u0.b);
          tma_prefetch_l2_4d(&tm_v, c * 64, u0.g, j * kBN, u0.b);
        }
    }
  }
  // A programmatic dependent launch: the prologue above touches only shared memory;
  // the previous kernel's writes are visible past this point, and TMEM is allocated
  // only after it (a kernel before this one may still hold TMEM on this SM).
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
  wc.set_limit(p.wait_limit_ns);
  wc.unit = 0;
  // The k-th unit of a reading warp (MMA or softmax): from the static deal, or from
  // the producer's queue entry k (false at the end of the work, or when the wait
  // gave up: `ok` is cleared then).
  auto next_unit = [&](int k, Unit& uu, bool& ok) -> bool {
    if (p.sched == nullptr) return unit_of<ALT>(p, k, uu);
    const int slot = k & (kUnitQueue - 1);
    if (!mbar_wait_warp(bar_uq_full(slot), (k / kUnitQueue) & 1u, wc, kSiteUnitQueue)) {
      ok = false;
      return false;
    }
    const int r = uq[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_uq_empty(slot));
    if (r < 0) return false;
    unit_from_rank<ALT>(p, r, uu);
    return true;
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;      // K/V slot loads issued
      uint32_t q_cnt = 0;   // Q loads issued
      bool ok = true;
      Unit u;
      // The producer's k-th unit: static, or the next rank of the global counter,
      // published in queue entry k for the other roles (-1: no more work).
      auto take_unit = [&](int k, Unit& uu) -> bool {
        if (p.sched == nullptr) return unit_of<ALT>(p, k, uu);
        const int slot = k & (kUnitQueue - 1);
        if (k >= kUnitQueue &&
            !mbar_wait_bounded(bar_uq_empty(slot), ((k / kUnitQueue) - 1) & 1u, wc, kSiteUnitQueue)) {
          ok = false;
          return false;
        }
        const unsigned r = atomicAdd(p.sched, 1u);
        const int rank = (r < static_cast<unsigned>(p.num_units)) ? static_cast<int>(r) : -1;
        uq[slot] = rank;
        mbar_arrive(bar_uq_full(slot));
        if (rank < 0) return false;
        unit_from_rank<ALT>(p, rank, uu);
        return true;
      };
      for (int k = 0; ok && take_unit(k, u); ++k) {
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
      // Every load of this CTA is issued: the next kernel on the stream may start (its
      // CTAs still wait for this grid's end before touching global memory or TMEM).
      asm volatile("griddepcontrol.launch_dependents;");
      // Whether or not this CTA aborted, the copies issued last may still be in
      // flight (another role can abort after this loop has ended, and then nothing
      // consumes them): let them land before the CTA can exit.
      for (uint32_t back = 1; back <= S && back <= it; ++back) {
        const uint32_t n = it - back;
        mbar_wait_drain(bar_full(n % S), (n / S) & 1u, wc, kSiteDrainLoads);
      }
      if (q_cnt > 0) mbar_wait_drain(bar_q_full, (q_cnt - 1) & 1u, wc, kSiteDrainLoads);
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ------------------------------------------------- MMA issuers, one per tile
    // Each tile has its own issuing warp, so one tile's MMAs never queue behind
    // the other tile's (tcgen05.mma issue blocks while the tensor core is busy).
    // The warp runs its loop warp-uniformly; one lane, picked by elect.sync,
    // issues each tcgen05 instruction.
    const int t = warp - kMmaWarp;
    constexpr uint32_t idesc_s = idesc_f16_f32acc(BF16, kBM, kBN, false);
    constexpr uint32_t idesc_o = idesc_f16_f32acc(BF16 && !kP16, kBM, D, true);
    // Descriptor bases. The start-address field holds (address >> 4) in its low
    // 14 bits; every operand address is below 256 KiB, so adding (offset >> 4)
    // to a base never carries out of that field.
    const uint64_t dq = sdesc_sw128(sQ + t * G::kTileBytes, 16, 1024);  // Q_t, K-major
    const uint64_t dk = sdesc_sw128(sKV, 16, 1024);                     // K slots, K-major
    const uint64_t dv = sdesc_sw128(sKV, G::kChunkBytes, 1024);         // V slots, MN-major
    const uint32_t mS = tmem_base + kColS0 + kStrideS * t;
    const uint32_t mP = tmem_base + kColP0 + kStrideP * t;
    const uint32_t mO = tmem_base + kColO0 + kStrideO * t;
    uint32_t it = 0, q_cnt = 0, p_cnt = 0, o_cnt = 0, ns = 0;
    bool ok = true;
    Unit u;
    auto slot_of = [&](uint32_t idx) { return idx % S; };
    auto par_of = [&](uint32_t idx) { return (idx / S) & 1u; };
    // S_t = Q_t · K_jᵀ from K slot `slot` (D/16 MMAs of K = 16), then commit s_full.
    auto issue_s = [&](uint32_t slot) __attribute__((always_inline)) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * G::kChunkBytes + (kk & 3) * 32;
        mma_ss_elect(mS, dq + (off >> 4), dk + ((slot * G::kTileBytes + off) >> 4), idesc_s,
                     kk > 0 ? 1u : 0u);
      }
      mma_commit_elect(bar_s_full(t));
      ++ns;
    };
    // O_t (+)= P_t · V_j from V slot `slot`. 16 keys per MMA: 8 TMEM columns of
    // packed P, 16 rows (2 KiB) of V. Split P keeps each 64-key half as
    // [hi 32 columns | lo 32 columns].
    auto issue_pv = [&](uint32_t slot, bool first, int kk_lo, int kk_hi) __attribute__((always_inline)) {
#pragma unroll
      for (int kk = kk_lo; kk < kk_hi; ++kk) {
        const uint32_t pcol = kSplitP ? (kk >> 2) * 64 + (kk & 3) * 8 : kk * 8;
        mma_ts_elect(mO, mP + pcol, dv + ((slot * G::kTileBytes + kk * 2048) >> 4), idesc_o,
                     (first && kk == 0) ? 0u : 1u);
      }
      if constexpr (kSplitP) {
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t pcol = (kk >> 2) * 64 + 32 + (kk & 3) * 8;
          mma_ts_elect(mO, mP + pcol, dv + ((slot * G::kTileBytes + kk * 2048) >> 4), idesc_o, 1u);
        }
      }
    };
    for (int k = 0; ok && next_unit(k, u, ok); ++k) {
      wc.unit = k;
      ok = mbar_wait_warp(bar_q_full, q_cnt & 1u, wc, kSiteMmaQFull);
      ++q_cnt;
      if (!ok) break;
      tc_fence_after();
      const uint32_t it0 = it;
      const TileSpan sp = (t == 0) ? u.t[0] : u.t[1];
      const bool live = sp.lo < sp.hi;
      const int j_lo = live ? sp.lo : u.hi, j_hi = live ? sp.hi : u.hi;
      auto kidx_of = [&](int j) { return it0 + 2u * (j - u.lo); };
      // Blocks of the unit this tile does not use: release their K and V slots,
      // but only once each load has landed — that proves the slot's previous
      // phase (both tiles' releases of its previous load) is complete, so this
      // release cannot be counted toward the wrong phase.
      auto skip_block = [&](int j) __attribute__((always_inline)) -> bool {
#pragma unroll
        for (uint32_t kv = 0; kv < 2; ++kv) {
          const uint32_t idx = kidx_of(j) + kv;
          if (!mbar_wait_warp(bar_full(slot_of(idx)), par_of(idx), wc, kSiteMmaKFull)) return false;
          if (lane == 0) mbar_arrive(bar_empty(slot_of(idx)));
          __syncwarp();
        }
        return true;
      };
      bool first = true;
      // O_t (+)= P_t(j) · V_j once P_t(j) is written; releases V_j's slot.
      auto pv_block = [&](int j) __attribute__((always_inline)) -> bool {
        const uint32_t vidx = kidx_of(j) + 1u;
        if (!mbar_wait_warp(bar_full(slot_of(vidx)), par_of(vidx), wc, kSiteMmaVFull)) return false;
        if constexpr (kHalves) {
          if (!mbar_wait_warp(bar_p_half(t), p_cnt & 1u, wc, kSiteMmaPFull)) return false;
        } else {
          if (!mbar_wait_warp(bar_p_full(t), p_cnt & 1u, wc, kSiteMmaPFull)) return false;
        }
        if (first && !mbar_wait_warp(bar_o_free(t), (o_cnt & 1u) ^ 1u, wc, kSiteMmaOFree))
          return false;
        tc_fence_after();
        if constexpr (kHalves) {
          issue_pv(slot_of(vidx), first, 0, kBN / 32);  // keys 0..63
          if (!mbar_wait_warp(bar_p_full(t), p_cnt & 1u, wc, kSiteMmaPFull)) return false;
          tc_fence_after();
          issue_pv(slot_of(vidx), false, kBN / 32, kBN / 16);  // keys 64..127
        } else {
          issue_pv(slot_of(vidx), first, 0, kBN / 16);
        }
        ++p_cnt;
        first = false;
        if constexpr (kSeparateP) mma_commit_elect(bar_pv_done(t));
        mma_commit_elect(bar_empty(slot_of(vidx)));
        return true;
      };
      if constexpr (ALT) {
        // This pipeline's blocks are lo + t, lo + t + 2, ...; the other pipeline's
        // blocks between them are released in order (skip_block).
        const int j_own = u.lo + t;
        const bool own = j_own < u.hi;
        auto s_block = [&](int j) __attribute__((always_inline)) -> bool {
          const uint32_t kidx = kidx_of(j);
          if (!mbar_wait_warp(bar_full(slot_of(kidx)), par_of(kidx), wc, kSiteMmaKFull)) return false;
          if (ns > 0 && !mbar_wait_warp(bar_s_free(t), (ns - 1) & 1u, wc, kSiteMmaSFree)) return false;
          tc_fence_after();
          issue_s(slot_of(kidx));
          mma_commit_elect(bar_empty(slot_of(kidx)));
          return true;
        };
        for (int j = u.lo; ok && j < (own ? j_own : u.hi); ++j) ok = skip_block(j);
        if (ok && own) {
          ok = s_block(j_own);
          for (int j = j_own; ok && j < u.hi; j += 2) {
            if (j + 1 < u.hi && !(ok = skip_block(j + 1))) break;
            if (j + 2 < u.hi && !(ok = s_block(j + 2))) break;
            ok = pv_block(j);
          }
          if (ok) {
            mma_commit_elect(bar_o_full(t));
            ++o_cnt;
          }
        }
        if (!ok) break;
        it = it0 + 2u * (u.hi - u.lo);
        mma_commit_elect(bar_q_free);
        continue;
      }
      for (int j = u.lo; ok && j < j_lo; ++j) ok = skip_block(j);
      if (ok && live) {
        if constexpr (kSeparateP) {
          // S_t(j+1) as soon as the softmax has read S_t(j) (s_free), then
          // O_t += P_t(j)·V_j: S, P and O have their own TMEM columns, so
          // S_t(j+1) overlaps the softmax of block j.
          auto s_block = [&](int j) __attribute__((always_inline)) -> bool {
            const uint32_t kidx = kidx_of(j);
            if (!mbar_wait_warp(bar_full(slot_of(kidx)), par_of(kidx), wc, kSiteMmaKFull))
              return false;
            if (ns > 0 && !mbar_wait_warp(bar_s_free(t), (ns - 1) & 1u, wc, kSiteMmaSFree))
              return false;
            tc_fence_after();
            issue_s(slot_of(kidx));
            mma_commit_elect(bar_empty(slot_of(kidx)));
            return true;
          };
          ok = s_block(j_lo);
          for (int j = j_lo; ok && j < j_hi; ++j) {
            if (j + 1 < j_hi && !(ok = s_block(j + 1))) break;
            ok = pv_block(j);
          }
        } else {
          // P over S: PV_t(j-1) is issued before S_t(j), which overwrites the
          // columns holding P_t; tcgen05 MMAs of one thread run in issue order.
          for (int j = j_lo; ok && j < j_hi; ++j) {
            const uint32_t kidx = kidx_of(j);
            ok = mbar_wait_warp(bar_full(slot_of(kidx)), par_of(kidx), wc, kSiteMmaKFull);
            if (ok && j > j_lo) ok = pv_block(j - 1);
            if (!ok) break;
            tc_fence_after();
            issue_s(slot_of(kidx));
            mma_commit_elect(bar_empty(slot_of(kidx)));
          }
          if (ok) ok = pv_block(j_hi - 1);
        }
        if (ok) {
          mma_commit_elect(bar_o_full(t));  // the tile's last P·V of this unit
          ++o_cnt;
        }
      }
      for (int j = j_hi; ok && j < u.hi; ++j) ok = skip_block(j);
      if (!ok) break;
      it = it0 + 2u * (u.hi - u.lo);
      mma_commit_elect(bar_q_free);
    }
    // Every MMA this warp issued has finished once the drain barrier flips
    // (both issuers commit to it).
    mma_commit_elect(bar_drain);
    mbar_wait_drain(bar_drain, 0, wc, kSiteMmaDrain);
  } else {
    // -------------------------------------------------------- softmax warps
    const int t = warp >> 2;
    const int quarter = warp & 3;
    const int r_in_tile = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem_base + lane_off + kColS0 + kStrideS * t;
    const uint32_t tP = tmem_base + lane_off + kColP0 + kStrideP * t;
    const uint32_t tO = tmem_base + lane_off + kColO0 + kStrideO * t;
    const float C = p.score_log2;
    uint32_t s_cnt = 0, o_cnt = 0;  // blocks / units this tile has processed (all units)
    [[maybe_unused]] uint32_t o1_cnt = 0, m_cnt = 0;  // ALT: tile 1's O_1 handed over, merges done
    bool ok = true;
    Unit u;
    for (int k = 0; ok && next_unit(k, u, ok); ++k) {
      wc.unit = k;
      const TileSpan span = (t == 0) ? u.t[0] : u.t[1];  // no dynamic index: stays in registers
      if (!ALT && span.lo >= span.hi) continue;
      // this tile's first block, and the step between its blocks
      const int j0 = ALT ? span.lo + t : span.lo;
      constexpr int kStep = ALT ? 2 : 1;
      const int row = span.row0 + r_in_tile;
      float m_ref = -INFINITY;  // reference max (base-2 units) the P values are relative to
      float l = 0.f;            // running sum of P
      // One key block; false when a wait gave up. Blocks that cross a mask boundary
      // run the masked instantiation in loops of their own before and after the
      // unmasked middle, so the hot loop holds one block body only (its code size
      // measurably matters: the masked body in the same loop cost 7 %).
      auto one_block = [&](int j, auto masked_tag) __attribute__((always_inline)) -> bool {
        constexpr bool masked = decltype(masked_tag)::value;
        if (!mbar_wait_warp(bar_s_full(t), s_cnt & 1u, wc, kSiteSmxSFull)) return false;
        tc_fence_after();
        const int key0 = j * kBN;
        int vis_lo = 0, vis_hi = kBN;  // visible columns of this row: [vis_lo, vis_hi)
        if constexpr (masked) {
          int hi_key = p.L;
          if (p.causal) hi_key = min(hi_key, row + 1);
          int lo_key = (p.window_left >= 0) ? row - p.window_left : 0;
          vis_hi = max(0, min(kBN, hi_key - key0));
          vis_lo = max(0, min(kBN, lo_key - key0));
        }
        // x = Cs · s with Cs = ±C, so that x carries the sign of the scale.
        const bool neg = p.negate_scores != 0;
        const float Cs = neg ? -C : C;
        float alpha = 1.f;
        bool rescale = false;
        bool stop = false;
        // The block body, instantiated twice: blocks that cross no mask boundary
        // (almost all of them) carry no per-element selects at all.
        auto block_body = [&](auto masked_tag) __attribute__((always_inline)) {
          constexpr bool M = decltype(masked_tag)::value;
          // One TMEM read of S (128 columns). S is released right away, the row
          // maximum and the exponentials both work from these registers.
          uint32_t sr[128];
          tmem_ld_x128(tS, sr);
          if constexpr (kSeparateP) {  // S is in registers: the next S MMA may overwrite it
            tc_fence_before();
            mbar_arrive(bar_s_free(t));
          }
          if constexpr (M) {  // masked keys: -inf for the max (+inf for the min), p = 0 below
            const uint32_t fill = neg ? 0x7f800000u : 0xff800000u;
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c < vis_lo || c >= vis_hi) sr[c] = fill;
          }
          float mx;  // max over visible columns of ±s (the sign of the scale)
          {
            float sv[128];
#pragma unroll
            for (int c = 0; c < 128; ++c) sv[c] = __uint_as_float(sr[c]);
            if (neg)
              mx = -row_min128(sv);
            else
              mx = row_max128(sv);
          }
          const float bm = (mx == -INFINITY) ? -INFINITY : mx * C;
          if (bm > m_ref + kThresh) {
            alpha = ex2_approx(m_ref - bm);  // 0 when m_ref is -inf
            m_ref = bm;
            rescale = true;
          }
          const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
          if constexpr (kSeparateP) {
            // P_t and O_t are read by this tile's previous P·V: wait until it is done.
            if (s_cnt > 0) {
              if (!mbar_wait_warp(bar_pv_done(t), (s_cnt - 1) & 1u, wc, kSiteSmxPvDone)) {
                stop = true;
                return;
              }
              tc_fence_after();
            }
          }
          // O rescale before the first half of this block's P·V (kHalves), once half
          // of the scores are consumed: 16 columns of O at a time.
          auto rescale_o_early = [&]() __attribute__((always_inline)) {
            if (__any_sync(0xffffffffu, rescale && j != j0)) {
              const float a = (rescale && j != j0) ? alpha : 1.f;
#pragma unroll 1
              for (int c0 = 0; c0 < D; c0 += 16) {
                uint32_t orow[16];
                tmem_ld_x16(tO + c0, orow);
#pragma unroll
                for (int c = 0; c < 16; ++c) orow[c] = __float_as_uint(__uint_as_float(orow[c]) * a);
                tmem_st_x16(tO + c0, orow);
              }
            }
          };
          const float2 c2 = make_float2(Cs, Cs);
          const float2 nmu2 = make_float2(-mu, -mu);
          float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          // P in 32-column chunks of 16 packed registers, stored to TMEM (P hi at
          // column c/2 of the P region; split P keeps each 64-key half h as
          // [hi 32 columns | lo 32 columns] at column 64h).
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t pk[16];
            uint32_t pk_lo[16];
            if constexpr (kF16Exp) {
              // Two exponentials per MUFU operation; the packed result is P.
              uint32_t prev = 0;
#pragma unroll
              for (int c = c0; c < c0 + 32; c += 2) {
                const float2 x = __ffma2_rn(
                    make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])),
                    make_float2(Cs, Cs), make_float2(-mu, -mu));
                __half2 xh = __floats2half2_rn(x.x, x.y);
                uint32_t pp = ex2_f16x2(*reinterpret_cast<uint32_t*>(&xh));
                if constexpr (M) {  // masked keys get exactly 0 (also when scale = 0)
                  const uint32_t keep = ((c >= vis_lo && c < vis_hi) ? 0x0000FFFFu : 0u) |
                                        ((c + 1 >= vis_lo && c + 1 < vis_hi) ? 0xFFFF0000u : 0u);
                  pp &= keep;
                }
                pk[(c - c0) >> 1] = pp;
                // row sum: two packed pairs added in fp16, then widened and
                // accumulated in fp32
                if ((c & 2) == 0) {
                  prev = pp;
                } else {
                  const __half2 s2 = __hadd2(*reinterpret_cast<__half2*>(&prev),
                                             *reinterpret_cast<__half2*>(&pp));
                  acc[(c >> 2) & 1] = __fadd2_rn(acc[(c >> 2) & 1], __half22float2(s2));
                }
              }
              tmem_st_x16(tP + (c0 >> 1), pk);
              if constexpr (kHalves) {
                if (c0 == 32) {  // keys 0..63 of P are stored: release them to the P·V
                  rescale_o_early();
                  tmem_st_wait();
                  tc_fence_before();
                  mbar_arrive(bar_p_half(t));
                }
              }
              continue;
            }
#pragma unroll
            for (int c = c0; c < c0 + 32; c += 2) {
              const float2 x = __ffma2_rn(
                  make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), c2, nmu2);
              const float x0 = x.x, x1 = x.y;
              float p0 = ex2_approx(x0);
              float p1 = ex2_approx(x1);
              if constexpr (M) {  // masked keys get exactly 0 (also when scale = 0)
                p0 = (c >= vis_lo && c < vis_hi) ? p0 : 0.f;
                p1 = (c + 1 >= vis_lo && c + 1 < vis_hi) ? p1 : 0.f;
              }
              acc[(c >> 1) & 1] = __fadd2_rn(acc[(c >> 1) & 1], make_float2(p0, p1));
              const uint32_t hi = pack2(p0, p1, kSplitP);  // bf16 halves or fp16 P
              pk[(c - c0) >> 1] = hi;
              if constexpr (kSplitP)
                pk_lo[(c - c0) >> 1] =
                    pack2(p0 - low_as_float(hi, BF16), p1 - high_as_float(hi, BF16), BF16);
            }
            if constexpr (kSplitP) {
              const int h = c0 >> 6, cl = c0 & 63;
              tmem_st_x16(tP + 64 * h + (cl >> 1), pk);
              tmem_st_x16(tP + 64 * h + 32 + (cl >> 1), pk_lo);
            } else {
              tmem_st_x16(tP + (c0 >> 1), pk);
            }
            if constexpr (kHalves) {
              if (c0 == 32) {
                rescale_o_early();
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar_p_half(t));
              }
            }
          }
          const float rowsum = (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
          l = l * alpha + rowsum;
        };
        block_body(masked_tag);
        if (stop) return false;
        ++s_cnt;
        // O rescale. The previous P·V of this tile is complete: with P over S,
        // S_t(j) was issued after it and s_full tracks all earlier MMAs; with a
        // separate P region, pv_done was waited just above.
        if (!kHalves && __any_sync(0xffffffffu, rescale && j != j0)) {
          const float a = (rescale && j != j0) ? alpha : 1.f;
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
        return true;
      };
      int ja, jb;
      unmasked_blocks(p, span, ja, jb);
      // the masked prefix, the unmasked middle (a tight loop of its own), the masked
      // suffix; one instance of each block body
      for (int j = j0; ok && j < span.hi;) {
        if (j >= ja && j < jb) {
          for (; ok && j < jb; j += kStep) ok = one_block(j, std::false_type{});
        } else {
          ok = one_block(j, std::true_type{});
          j += kStep;
        }
      }
      if (!ok) break;
      if constexpr (ALT) {
        if (t == 1) {
          // hand this row's max and sum to tile 0, which reads O_1 from TMEM
          if (m_cnt > 0 && !mbar_wait_warp(bar_merge_free, (m_cnt - 1) & 1u, wc, kSiteSmxOFull)) break;
          xchg[r_in_tile] = make_float2(m_ref, l);
          mbar_arrive(bar_merge_ready);
          ++m_cnt;
          continue;
        }
      }
      // ---- epilogue: O / l and LSE for this tile
      ok = mbar_wait_warp(bar_o_full(t), o_cnt & 1u, wc, kSiteSmxOFull);
      ++o_cnt;
      if (!ok) break;
      [[maybe_unused]] bool live1 = false;
      [[maybe_unused]] float w0 = 1.f, w1 = 0.f;
      if constexpr (ALT) {
        // combine with tile 1's part: its max and sum from shared memory, O_1 from TMEM
        live1 = span.lo + 1 < span.hi;
        if (!(ok = mbar_wait_warp(bar_merge_ready, m_cnt & 1u, wc, kSiteSmxOFull))) break;
        if (live1) {
          if (!(ok = mbar_wait_warp(bar_o_full(1), o1_cnt & 1u, wc, kSiteSmxOFull))) break;
          ++o1_cnt;
        }
        const float2 ml1 = xchg[r_in_tile];
        const float mm = fmaxf(m_ref, ml1.x);
        w0 = (l > 0.f) ? ex2_approx(m_ref - mm) : 0.f;
        w1 = (ml1.y > 0.f) ? ex2_approx(ml1.x - mm) : 0.f;
        l = l * w0 + ml1.y * w1;
        m_ref = mm;
      }
      tc_fence_after();
      // Opaque copies: keep the compiler from hoisting the epilogue's 64-bit
      // addresses above the block loop, where they would hold registers the
      // softmax needs.
      int eb = u.b, eh = u.h, erow = row;
      asm volatile("" : "+r"(eb), "+r"(eh), "+r"(erow));
      const bool live = erow < p.L;
      float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      if constexpr (PV16) inv_l *= exp2_int(-v16_exponent(p.vmax[eb * p.Hkv + eh / (p.Hq / p.Hkv)]));
      const size_t o_row = ((static_cast<size_t>(eb) * p.L + erow) * p.Hq + eh) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t orow[32];
        tmem_ld_x32(tO + c0, orow);
        if constexpr (ALT) {
          uint32_t o1[32];
          tmem_ld_x32(tO + kStrideO + c0, o1);  // O_1: the same lanes, tile 1's columns
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float a = __uint_as_float(orow[c]) * w0;
            orow[c] = __float_as_uint(w1 > 0.f ? a + __uint_as_float(o1[c]) * w1 : a);
          }
        }
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
        p.lse[(static_cast<size_t>(eb) * p.Hq + eh) * p.L + erow] = lse;
      }
      tc_fence_before();
      mbar_arrive(bar_o_free(t));
      if constexpr (ALT) {
        if (live1) mbar_arrive(bar_o_free(1));  // O_1 has been read
        mbar_arrive(bar_merge_free);
        ++m_cnt;
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

}  // namespace ex19
