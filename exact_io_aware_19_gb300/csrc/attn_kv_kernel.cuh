// attn_kv_kernel.cuh — decode-shaped (split-KV) exact attention forward for sm_103a.
//
// What it computes: the attention of the square kernel for Lq query rows that are
// the last Lq positions of an Lk-long sequence (row i sits at position
// Lk - Lq + i; causal and window masks are taken at that position). Row p sees
// keys [p - window_left, p + window_right] (each bound -1 = none; causal is the
// right bound 0), the window_size = (left, right) option of the "Flash Attention
// optimization" skill page (workflow 2 step 3). This is a
// generation step reading the whole KV cache, the case "What is memory-efficient
// attention for long context on 8x H100?" (section 1, key limitations) names as
// bound by HBM bandwidth. The keys of a row tile may be cut into `splits`
// consecutive ranges computed by different CTAs; each writes its partial O / l
// and log2-sum-exp, and attn_kv_merge_kernel combines them by their log-sum-exp
// (attention computed in parts, same page, section 4).
//
// GB300 mapping (one CTA per (batch, K/V head, row tile, key split)):
//   * The `group` query heads that read one K/V head are packed into the rows of
//     one 128-row tile: row r of the tile is query position i0 + r / group, head
//     g * group + r % group. One TMA box {64 of d, group heads, q_per_tile rows}
//     lands the tile in shared memory in exactly that order, so K and V stream
//     once per group instead of once per query head.
//   * warp 8 (producer): TMA loads of Q and of K_j, V_j into a ring of slots.
//   * warp 9 (MMA): one elected lane issues every tcgen05.mma. Block j's
//     S = Q K_jᵀ goes to TMEM buffer j mod 2 (128 fp32 columns); the softmax
//     writes P over the scores it has read (keys 64h .. 64h + 63 of half h from
//     column 64h); O += P V_j reads P back from there.
//     S(j + 2) is issued after P·V(j), so buffer reuse needs no barrier (MMAs of
//     one thread run in issue order), and S(j + 1) runs under the softmax of j.
//   * warps 0-7 (softmax): two threads per tile row. Warp w reads TMEM lanes
//     32 (w mod 4) .. + 31 and the key half w / 4 (64 of the block's 128 scores),
//     so each SM sub-partition runs two softmax warps with half a row's work each.
//     The two halves of a row trade their partial maxima through shared memory
//     (an mbarrier per warp pair and buffer, bounded waits) and both take the same
//     reference max; each keeps its own running sum l, P = 2^(x - m) for its keys
//     and the O rescale of its half of the columns; the halves' sums meet once in
//     the epilogue, which writes O / l and the log-sum-exp.
//   * Paged K/V cache ("What is memory-efficient attention ...", section 3: the
//     cache is cut into fixed-size blocks of tokens stored anywhere, and a page
//     table maps each sequence's logical blocks to physical pages): a 128-key block
//     is fetched as 128 / page_size TMA boxes of page_size rows, one per page, each
//     landing at its row offset of the slot (the 128-byte swizzle depends only on
//     the shared-memory address, so the pieces form the same tile as one box).
//     Each sequence has its own length. Pages past its end, and table entries
//     outside [0, num_pages), are fetched at an out-of-range row, which TMA fills
//     with zeros. The unused rows of a partial last page hold whatever the cache
//     holds, so the MMA warp zeroes those V rows in shared memory before that
//     block's P·V (P is 0 there, but 0 · NaN would not be).
//     The paged producer is the whole warp: its lanes hold the page rows of the next
//     32 / (128 / page_size) blocks, loaded a window ahead, and lane pp issues page
//     pp's copies, so neither page-table latency nor a serial issue of small boxes
//     paces the stream.
//   * Items of at most 32 query rows (a decode step) run the keys-on-lanes kernel of
//     attn_kv_keys_kernel.cuh instead, with the same items, splits and partials.
//   * Every wait is bounded; a timeout sets the status word and all roles leave.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <type_traits>

#include "attn_kv_params.h"
#include "row_ops.cuh"
#include "sm103_ptx.cuh"
#include "tmem_io.cuh"
#include "vscale.cuh"

namespace ex19 {
namespace kv {

constexpr int kBM = 128;             // rows per tile (= TMEM lanes)
constexpr int kBN = 128;             // keys per K/V block

// Warp roles and TMEM columns.
struct KvRoles {
  static constexpr int kSmxWarps = 8;                          // softmax warps (two per lane quarter)
  static constexpr int kHalves = 2;                            // softmax threads per row
  static constexpr int kThreads = 32 * (kSmxWarps + 2);        // + producer warp + MMA warp
  static constexpr int kProducerWarp = kSmxWarps;
  static constexpr int kMmaWarp = kSmxWarps + 1;
  static constexpr uint32_t kTmemCols = 512;
  // S0 [0,128), S1 [128,256) with P over them, O [256, 256 + D)
  static constexpr uint32_t kColO = 256;
};

enum : uint32_t {
  kSiteProdEmpty = 0x50001,
  kSiteMmaQFull = 0x60001, kSiteMmaKFull = 0x60002, kSiteMmaVFull = 0x60003,
  kSiteMmaPFull = 0x60004, kSiteMmaDrain = 0x60005,
  kSiteSmxSFull = 0x70001, kSiteSmxOFull = 0x70002, kSiteSmxPvDone = 0x70003,
  kSiteSmxExchange = 0x70004,
  kSiteDrainLoads = 0x80001,
  kSiteBadSeqLen = 0x90001,  // a paged sequence length outside [Lq, max_seq_len]
};

template <int D>
struct KvGeometry {
  static constexpr int kChunks = D / 64;          // 128-byte swizzle boxes per row
  static constexpr int kChunkBytes = kBM * 128;   // one box column of a 128-row tile
  static constexpr int kTileBytes = kBM * D * 2;  // a 128-row tile of Q, K or V
  static constexpr int kSlots = (D == 64) ? 8 : 5;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kTileBytes;
  static constexpr int kOffBar = kOffKV + kSlots * kTileBytes;
  // barriers: full[S], empty[S], q_full, s_full[2], p_full[2], pv_done[2], o_full,
  // drain, exchange[4 warp pairs][2 buffers]
  static constexpr int kNumBars = 2 * kSlots + 17;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
  // the two halves of a row trade one float per round: [2 buffers][2 halves][128 rows]
  static constexpr int kOffX = kOffMisc + 16;
  static constexpr int kXBytes = 2 * 2 * kBM * 4;
  static constexpr int kSmemUsed = kOffX + kXBytes;
  static constexpr int kSmemBytes = kSmemUsed + 1024;     // slack to align the base to 1024
};

// The work item of this CTA and its key blocks [lo, hi).
struct KvItem {
  int b, g, split;
  int i0, i1;  // query positions [i0, i1) of the tile
  int lo, hi;  // key blocks of this split
  int Lk;      // keys of this batch entry's sequence
  bool bad;    // paged: the sequence length is out of range (nothing is computed)
};

// Maximum of a 64-value half row: 8 independent chains (8 values each, 3-input
// maxima), then a tree.
__device__ __forceinline__ float row_max64(const float (&s)[64]) {
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a = max3f(s[i], s[8 + i], s[16 + i]);
    a = max3f(a, s[24 + i], s[32 + i]);
    a = max3f(a, s[40 + i], s[48 + i]);
    m[i] = fmaxf(a, s[56 + i]);
  }
  return fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])), fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
}

// Minimum of a 64-value half row (used when the scale is negative).
__device__ __forceinline__ float row_min64(const float (&s)[64]) {
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a = s[i];
#pragma unroll
    for (int k = 8; k < 64; k += 8) a = fminf(a, s[k + i]);
    m[i] = a;
  }
  return fminf(fminf(fminf(m[0], m[1]), fminf(m[2], m[3])), fminf(fminf(m[4], m[5]), fminf(m[6], m[7])));
}

// Right bound of a row's visible keys relative to its position (-1: none).
__device__ __forceinline__ int right_bound(const KvParams& p) { return p.causal ? 0 : p.window_right; }

template <bool PAGED>
__device__ __forceinline__ KvItem kv_item(const KvParams& p) {
  KvItem it;
  // CTA order: row tile outermost and descending (under a causal mask the last row
  // tiles see the most keys), then (batch, K/V head), then split, so that the CTAs
  // with the most work start first and the short ones fill the end of the grid
  int x = blockIdx.x;
  it.split = x % p.splits;
  x /= p.splits;
  const int nbg = p.B * p.Hkv;
  const int rt = p.row_tiles - 1 - x / nbg;
  x %= nbg;
  it.g = x % p.Hkv;
  it.b = x / p.Hkv;
  it.i0 = rt * p.q_per_tile;
  it.i1 = min(p.Lq, it.i0 + p.q_per_tile);
  it.Lk = p.Lk;
  it.bad = false;
  if constexpr (PAGED) {
    it.Lk = p.seq_lens[it.b];
    if (it.Lk < p.Lq || it.Lk > p.Lk) {
      it.bad = true;
      it.Lk = p.Lq;
    }
  }
  const int off = it.Lk - p.Lq;  // position of query row 0
  const int nblk = (it.Lk + kBN - 1) / kBN;
  const int wr = right_bound(p);
  const int blk_hi = (wr >= 0) ? min(nblk, (off + it.i1 - 1 + wr) / kBN + 1) : nblk;
  const int blk_lo = (p.window_left >= 0) ? max(0, off + it.i0 - p.window_left) / kBN : 0;
  const long long n = blk_hi - blk_lo;
  it.lo = blk_lo + static_cast<int>(n * it.split / p.splits);
  it.hi = blk_lo + static_cast<int>(n * (it.split + 1) / p.splits);
  if (it.bad) it.hi = it.lo;
  return it;
}

// Asks for the first `nblk` key blocks of a dense-cache work item (K and V) in L2,
// before griddepcontrol.wait: a prefetch is only a hint, so the loads after the wait
// still read what the kernels before this one left (their stores reach L2 as well).
// The work item of a dense cache needs no global read.
template <int D>
__device__ __forceinline__ void kv_prefetch_first_blocks(const KvParams& p, const CUtensorMap* tm_k,
                                                         const CUtensorMap* tm_v, int nblk) {
  const KvItem it0 = kv_item<false>(p);
  for (int j = it0.lo; j < min(it0.hi, it0.lo + nblk); ++j)
    for (int c = 0; c < D / 64; ++c) {
      tma_prefetch_l2_4d(tm_k, c * 64, it0.g, j * kBN, it0.b);
      tma_prefetch_l2_4d(tm_v, c * 64, it0.g, j * kBN, it0.b);
    }
}

// The TMA producer warp of the one-tile kernels: the Q tile of the work item, then K_j
// and V_j of its blocks [it.lo, it.hi) into a ring of S slots of 128 keys × D (slot s
// at sKV + s·128·D·2; its full barrier at bars + 8s, its empty barrier at bars +
// 8(S + s)); q_full at bars + 16S. Q chunk c (64 columns) lands at sQ + c·q_chunk_bytes.
// The whole warp calls it (the paged producer uses every lane).
template <bool PAGED, int D>
__device__ __forceinline__ void kv_produce(const KvParams& p, const KvItem& it, int nblocks,
                                           const CUtensorMap* tm_q_, const CUtensorMap* tm_k_,
                                           const CUtensorMap* tm_v_, uint32_t sQ,
                                           uint32_t q_chunk_bytes, uint32_t sKV, int S,
                                           uint32_t bars, const WaitCtl& wc, int lane) {
  constexpr int kChunks = D / 64;
  constexpr int kTileBytes = kBM * D * 2;
  constexpr int kChunkBytes = kBM * 128;
  auto bar_full = [&](uint32_t s) { return bars + 8u * s; };
  auto bar_empty = [&](uint32_t s) { return bars + 8u * (S + s); };
  const uint32_t bar_q_full = bars + 8u * (2 * S);
  const CUtensorMap& tm_q = *tm_q_;
  const CUtensorMap& tm_k = *tm_k_;
  const CUtensorMap& tm_v = *tm_v_;
  if (nblocks > 0) {
    if (lane == 0) {
      // The Q box is {64, group, q_per_tile, 1}; rows past Lq are zero-filled and
      // still counted in the transaction bytes.
      mbar_arrive_expect_tx(bar_q_full, kChunks * 128u * p.group * p.q_per_tile);
      for (int c = 0; c < kChunks; ++c)
        tma_load_4d(sQ + c * q_chunk_bytes, &tm_q, bar_q_full, c * 64, it.g * p.group, it.i0,
                    it.b);
    }
    uint32_t n = 0;
    bool ok = true;
    if constexpr (PAGED) {
      // The whole warp runs the loop: its 32 lanes hold the physical rows of the
      // pages of a window of W = 32 / P blocks (P = 128 / page_size pages per block),
      // and the next window's page-table loads are issued when the current window
      // starts, so they land long before they are needed (a table read per block,
      // right before its TMA, put an L2 round trip under load on every block).
      // Lane 0 takes each page's row by shuffle and issues the copies.
      const int P = kBN / p.page_size;
      const int W = 32 / P;
      const int oob_row = p.num_pages * p.page_size;  // past the cache: zero-filled
      auto fetch = [&](int j0) -> int {  // this lane's page of the window starting at j0
        const int jb = j0 + lane / P, lp = jb * P + lane % P;  // block, logical page
        int phys = -1;
        if (jb < it.hi && lp * p.page_size < it.Lk)
          phys = p.block_table[static_cast<size_t>(it.b) * p.max_pages + lp];
        return (phys >= 0 && phys < p.num_pages) ? phys * p.page_size : oob_row;
      };
      int cur = fetch(it.lo), nxt = oob_row;
      for (int j = it.lo; ok && j < it.hi; ++j) {
        const int jw = (j - it.lo) % W;
        if (jw == 0) nxt = fetch(j + W);
        for (int kv = 0; ok && kv < 2; ++kv) {
          const uint32_t slot = n % S;
          ok = mbar_wait_warp(bar_empty(slot), ((n / S) & 1u) ^ 1u, wc, kSiteProdEmpty);
          if (!ok) break;
          if (lane == 0) mbar_arrive_expect_tx(bar_full(slot), kTileBytes);
          __syncwarp();  // the transaction count is set before any copy can complete
          const CUtensorMap* tm = kv ? &tm_v : &tm_k;
          // lane pp < P copies page pp of this block: one box of page_size rows
          const int row = __shfl_sync(0xffffffffu, cur, jw * P + (lane % P));
          if (lane < P) {
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
              tma_load_4d(sKV + slot * kTileBytes + c * kChunkBytes + lane * p.page_size * 128,
                          tm, bar_full(slot), c * 64, it.g, row, 0);
          }
          ++n;
        }
        if (jw == W - 1) cur = nxt;
      }
    } else if (lane == 0) {
      for (int j = it.lo; ok && j < it.hi; ++j) {
        for (int kv = 0; kv < 2; ++kv) {
          const uint32_t slot = n % S;
          ok = mbar_wait_bounded(bar_empty(slot), ((n / S) & 1u) ^ 1u, wc, kSiteProdEmpty);
          if (!ok) break;
          mbar_arrive_expect_tx(bar_full(slot), kTileBytes);
          const CUtensorMap* tm = kv ? &tm_v : &tm_k;
          for (int c = 0; c < kChunks; ++c)
            tma_load_4d(sKV + slot * kTileBytes + c * kChunkBytes, tm, bar_full(slot),
                        c * 64, it.g, j * kBN, it.b);
          ++n;
        }
      }
    }
    if (lane == 0) {
      // Whether or not this CTA aborted, the copies issued last may still be in
      // flight (another role can abort after this loop has ended, and then nothing
      // consumes them): let them land before the CTA can exit.
      for (uint32_t back = 1; back <= S && back <= n; ++back) {
        const uint32_t m = n - back;
        mbar_wait_drain(bar_full(m % S), (m / S) & 1u, wc, kSiteDrainLoads);
      }
      mbar_wait_drain(bar_q_full, 0, wc, kSiteDrainLoads);
    }
  }
}

// PV16 (bf16 inputs only): V is the call's fp16 copy scaled per (batch, K/V head)
// by 2^e (vscale.cuh), P is fp16 and P·V one fp16 product; the output is scaled back.
template <int D, bool BF16, bool OUT_F32, bool PAGED, bool PV16 = false>
__global__ void __launch_bounds__(KvRoles::kThreads, 1)
    attn_kv_sm103_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const KvParams p) {
  using G = KvGeometry<D>;
  using R = KvRoles;
  constexpr int kProducerWarp = R::kProducerWarp;
  constexpr int kMmaWarp = R::kMmaWarp;
  constexpr uint32_t kTmemCols = R::kTmemCols;
  constexpr uint32_t kColO = R::kColO;
  constexpr int S = G::kSlots;
  static_assert(!PV16 || (BF16 && !PAGED), "the fp16 copy of V is for dense bfloat16 inputs");
  constexpr bool kSplitP = BF16 && !PV16;  // bf16 P as hi + lo halves (two P·V MMAs)
  constexpr bool kF16Exp = !BF16;  // fp16 inputs: exponentials on packed fp16 pairs
  constexpr float kThresh = kF16Exp ? 1.0f : 8.0f;  // log2 units of max growth before a rescale

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
  auto bar_s_full = [&](uint32_t b) { return bars + 8u * (2 * S + 1 + b); };
  auto bar_p_full = [&](uint32_t b) { return bars + 8u * (2 * S + 3 + b); };
  auto bar_pv_done = [&](uint32_t b) { return bars + 8u * (2 * S + 5 + b); };
  const uint32_t bar_o_full = bars + 8u * (2 * S + 7);
  const uint32_t bar_drain = bars + 8u * (2 * S + 8);
  // exchange between the two softmax warps of lane quarter q, buffer b
  auto bar_x = [&](int q, uint32_t b) { return bars + 8u * (2 * S + 9 + 2 * q + b); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + G::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Prologue: shared memory and the tensor maps only (no global memory, no TMEM),
  // so it may overlap the previous kernel on the stream.
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_q_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_s_full(b), 1);
      mbar_init(bar_p_full(b), R::kSmxWarps * 32);
      mbar_init(bar_pv_done(b), 1);
    }
    mbar_init(bar_o_full, 1);
    mbar_init(bar_drain, 1);
    for (int q = 0; q < 4; ++q)
      for (uint32_t b = 0; b < 2; ++b) mbar_init(bar_x(q, b), 64);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    if constexpr (!PAGED && !kSplitP) kv_prefetch_first_blocks<D>(p, &tm_k, &tm_v, 4);
  }
  // Launched as a programmatic dependent: past this point the previous kernel's
  // writes (Q, K, V, the page table, a merge still reading this workspace) are
  // complete and visible. TMEM is allocated only after it, so this CTA never holds
  // TMEM while it waits on a kernel that may still need some. A no-op for an
  // ordinary launch.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const KvItem it = kv_item<PAGED>(p);
  const int nblocks = max(0, it.hi - it.lo);

  WaitCtl wc;
  wc.abort_flag = abort_flag;
  wc.status = p.status;
  wc.set_limit(p.wait_limit_ns);
  wc.unit = blockIdx.x;
  if (it.bad) {
    // Nothing of this batch entry is computed or written; report it once per CTA.
    if (threadIdx.x == 0) record_error(wc, kStatusInvalidArg, kSiteBadSeqLen);
  }

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    kv_produce<PAGED, D>(p, it, nblocks, &tm_q, &tm_k, &tm_v, sQ, G::kChunkBytes, sKV, S, bars, wc,
                         lane);
    // Every load of this CTA has landed: the next kernel on the stream may start (its
    // CTAs still wait for this grid's end before touching global memory or TMEM).
    // Not when a merge kernel follows (it measured slower launched early).
    if (p.splits <= 1 && lane == 0) asm volatile("griddepcontrol.launch_dependents;");
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA issuer
    if (nblocks > 0) {
      constexpr uint32_t idesc_s = idesc_f16_f32acc(BF16, kBM, kBN, false);
      constexpr uint32_t idesc_o = idesc_f16_f32acc(kSplitP, kBM, D, true);
      const uint64_t dq = sdesc_sw128(sQ, 16, 1024);               // Q tile, K-major
      const uint64_t dk = sdesc_sw128(sKV, 16, 1024);              // K slots, K-major
      const uint64_t dv = sdesc_sw128(sKV, G::kChunkBytes, 1024);  // V slots, MN-major
      const uint32_t mO = tmem_base + kColO;
      auto slot_of = [&](uint32_t idx) { return idx % S; };
      auto par_of = [&](uint32_t idx) { return (idx / S) & 1u; };
      // S = Q · K_jᵀ (block jj of the split) into buffer jj & 1; releases K_j.
      auto issue_s = [&](int jj) __attribute__((always_inline)) -> bool {
        const uint32_t kidx = 2u * jj;
        if (!mbar_wait_warp(bar_full(slot_of(kidx)), par_of(kidx), wc, kSiteMmaKFull)) return false;
        tc_fence_after();
        const uint32_t mS = tmem_base + 128u * (jj & 1);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * G::kChunkBytes + (kk & 3) * 32;
          mma_ss_elect(mS, dq + (off >> 4), dk + ((slot_of(kidx) * G::kTileBytes + off) >> 4),
                       idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit_elect(bar_s_full(jj & 1));
        mma_commit_elect(bar_empty(slot_of(kidx)));
        return true;
      };
      // O (+)= P · V_j once the softmax has written P into buffer jj & 1; releases V_j.
      auto issue_pv = [&](int jj) __attribute__((always_inline)) -> bool {
        const uint32_t vidx = 2u * jj + 1u;
        if (!mbar_wait_warp(bar_full(slot_of(vidx)), par_of(vidx), wc, kSiteMmaVFull)) return false;
        if constexpr (PAGED) {
          // Rows past the sequence in its last block: the part of a partial page
          // the TMA did load holds arbitrary cache contents; make every such V row 0.
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
        if (!mbar_wait_warp(bar_p_full(jj & 1), (jj >> 1) & 1u, wc,
                            kSiteMmaPFull))
          return false;
        tc_fence_after();
        const uint32_t mP = tmem_base + 128u * (jj & 1);
        const uint64_t dvs = dv + ((slot_of(vidx) * G::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // keys 16 kk .. 16 kk + 15: each
          // 64-key half h sits at column 64 h (bf16: hi there, lo 32 columns on)
          const uint32_t pcol = (kk >> 2) * 64 + (kk & 3) * 8;
          mma_ts_elect(mO, mP + pcol, dvs + ((kk * 2048) >> 4), idesc_o,
                       (jj == 0 && kk == 0) ? 0u : 1u);
        }
        if constexpr (kSplitP) {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint32_t pcol = (kk >> 2) * 64 + 32 + (kk & 3) * 8;
            mma_ts_elect(mO, mP + pcol, dvs + ((kk * 2048) >> 4), idesc_o, 1u);
          }
        }
        mma_commit_elect(bar_pv_done(jj & 1));
        mma_commit_elect(bar_empty(slot_of(vidx)));
        return true;
      };
      bool ok = mbar_wait_warp(bar_q_full, 0, wc, kSiteMmaQFull);
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
    // Every MMA this warp issued has finished once the drain barrier flips.
    mma_commit_elect(bar_drain);
    mbar_wait_drain(bar_drain, 0, wc, kSiteMmaDrain);
  } else {
    // -------------------------------------------------------- softmax warps
    constexpr int kHalves = R::kHalves;
    constexpr int kCols = kBN / kHalves;  // scores of a block per softmax thread
    constexpr int kOCols = D / kHalves;   // O columns this thread rescales and writes
    const int quarter = warp & 3;         // TMEM lane quarter of this warp
    const int ch = warp >> 2;             // key half of this warp
    const int col0 = ch * kCols;          // first score column of this thread
    const int rho = quarter * 32 + lane;  // row of the tile
    const bool row_ok = !it.bad && rho < (it.i1 - it.i0) * p.group;
    const int qi = it.i0 + rho / p.group;  // query position (may be >= Lq for unused rows)
    const int h = it.g * p.group + rho % p.group;
    const int Lk = it.Lk;
    const int off = Lk - p.Lq;
    const int pos = off + qi;
    const int pos_min = off + it.i0, pos_max = off + it.i1 - 1;
    const int wr = right_bound(p);
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tO = tmem_base + lane_off + kColO;
    const float C = p.score_log2;
    const bool neg = p.negate_scores != 0;
    const float Cs = neg ? -C : C;  // x = Cs · s carries the sign of the scale
    float m_ref = -INFINITY;        // reference max (base-2 units), the same in both halves
    float l = 0.f;                  // running sum of this thread's P
    bool ok = true;
    // Round n of the two halves of a row: each stores its value, arrives on the
    // pair's barrier of buffer n mod 2 and, once both have, reads the other's. A
    // buffer is written again two rounds later, after the round in between has
    // completed, which needs the other half's arrival, made after its read.
    float* xbuf = reinterpret_cast<float*>(smem + G::kOffX);
    auto exchange = [&](uint32_t n, float v, float& other) -> bool {
      const uint32_t b = n & 1u;
      xbuf[(b * 2 + ch) * kBM + rho] = v;
      mbar_arrive(bar_x(quarter, b));
      if (!mbar_wait_warp(bar_x(quarter, b), (n >> 1) & 1u, wc, kSiteSmxExchange)) return false;
      other = xbuf[(b * 2 + (ch ^ 1)) * kBM + rho];
      return true;
    };
    // One key block (jj-th of this CTA); false when a wait gave up. Blocks that cross
    // a mask boundary run the masked instantiation outside the unmasked middle's own
    // tight loop, so the hot loop holds one block body only.
    auto one_block = [&](int jj, auto masked_tag) __attribute__((always_inline)) -> bool {
      constexpr bool masked = decltype(masked_tag)::value;
      const int j = it.lo + jj;
      const uint32_t buf = jj & 1;
      if (!mbar_wait_warp(bar_s_full(buf), (jj >> 1) & 1u, wc, kSiteSmxSFull))
        return false;
      tc_fence_after();
      // S of this block, then P over the scores this thread has read
      const uint32_t tS = tmem_base + lane_off + 128u * buf;
      const uint32_t tP = tS;
      const int key0 = j * kBN;
      int vis_lo = 0, vis_hi = kBN;  // visible columns of this row: [vis_lo, vis_hi)
      if constexpr (masked) {
        const int hi_key = (wr >= 0) ? min(Lk, pos + wr + 1) : Lk;
        const int lo_key = (p.window_left >= 0) ? pos - p.window_left : 0;
        vis_hi = max(0, min(kBN, hi_key - key0));
        vis_lo = max(0, min(kBN, lo_key - key0));
      }
      float alpha = 1.f;
      bool rescale = false;
      bool stop = false;
      auto block_body = [&](auto masked_tag) __attribute__((always_inline)) {
        constexpr bool M = decltype(masked_tag)::value;
        uint32_t sr[kCols];
        tmem_ld_x64(tS + col0, sr);
        if constexpr (M) {  // masked keys: -inf for the max (+inf for the min), p = 0 below
          const uint32_t fill = neg ? 0x7f800000u : 0xff800000u;
#pragma unroll
          for (int c = 0; c < kCols; ++c)
            if (col0 + c < vis_lo || col0 + c >= vis_hi) sr[c] = fill;
        }
        float mx;
        {
          float sv[kCols];
#pragma unroll
          for (int c = 0; c < kCols; ++c) sv[c] = __uint_as_float(sr[c]);
          mx = neg ? -row_min64(sv) : row_max64(sv);
        }
        if constexpr (kHalves == 2) {
          // the row max over both halves, combined in the same order by both
          float other;
          if (!exchange(static_cast<uint32_t>(jj), mx, other)) {
            stop = true;
            return;
          }
          mx = (ch == 0) ? fmaxf(mx, other) : fmaxf(other, mx);
        }
        const float bm = (mx == -INFINITY) ? -INFINITY : mx * C;
        if (bm > m_ref + kThresh) {
          alpha = ex2_approx(m_ref - bm);  // 0 when m_ref is -inf
          m_ref = bm;
          rescale = true;
        }
        const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
        float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c0 = 0; c0 < kCols; c0 += 32) {
          uint32_t pk[16];
          [[maybe_unused]] uint32_t pk_lo[16];  // bf16: the low halves of split P
          [[maybe_unused]] uint32_t prev = 0;   // fp16: the pair summed with the next
#pragma unroll
          for (int c = c0; c < c0 + 32; c += 2) {
            const int cg = col0 + c;  // column within the block
            const float2 x = __ffma2_rn(
                make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])),
                make_float2(Cs, Cs), make_float2(-mu, -mu));
            if constexpr (kF16Exp) {
              __half2 xh = __floats2half2_rn(x.x, x.y);
              uint32_t pp = ex2_f16x2(*reinterpret_cast<uint32_t*>(&xh));
              if constexpr (M) {  // masked keys get exactly 0 (also when scale = 0)
                const uint32_t keep = ((cg >= vis_lo && cg < vis_hi) ? 0x0000FFFFu : 0u) |
                                      ((cg + 1 >= vis_lo && cg + 1 < vis_hi) ? 0xFFFF0000u : 0u);
                pp &= keep;
              }
              pk[(c - c0) >> 1] = pp;
              if ((c & 2) == 0) {
                prev = pp;
              } else {  // two packed pairs summed in fp16, then accumulated in fp32
                const __half2 s2 = __hadd2(*reinterpret_cast<__half2*>(&prev),
                                           *reinterpret_cast<__half2*>(&pp));
                acc[(c >> 2) & 1] = __fadd2_rn(acc[(c >> 2) & 1], __half22float2(s2));
              }
            } else {
              float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
              if constexpr (M) {
                p0 = (cg >= vis_lo && cg < vis_hi) ? p0 : 0.f;
                p1 = (cg + 1 >= vis_lo && cg + 1 < vis_hi) ? p1 : 0.f;
              }
              acc[(c >> 1) & 1] = __fadd2_rn(acc[(c >> 1) & 1], make_float2(p0, p1));
              const uint32_t hi = pack2(p0, p1, kSplitP);  // bf16 halves or fp16 P
              pk[(c - c0) >> 1] = hi;
              if constexpr (kSplitP)
                pk_lo[(c - c0) >> 1] =
                    pack2(p0 - low_as_float(hi, BF16), p1 - high_as_float(hi, BF16), BF16);
            }
          }
          // P of keys [64 hh, 64 hh + 64) at column 64 hh, over scores this thread has
          // already read; split P keeps
          // [hi 32 columns | lo 32 columns] there.
          const int cb = col0 + c0;  // first key of this chunk
          if constexpr (kSplitP) {
            const int hh = cb >> 6, cl = cb & 63;
            tmem_st_x16(tP + 64 * hh + (cl >> 1), pk);
            tmem_st_x16(tP + 64 * hh + 32 + (cl >> 1), pk_lo);
          } else {
            tmem_st_x16(tP + 64 * (cb >> 6) + ((cb & 63) >> 1), pk);
          }
        }
        l = l * alpha + ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y));
      };
      block_body(masked_tag);
      if (stop) return false;
      // O rescale (this thread's columns) once the previous P·V, which accumulates
      // into O, is complete; the first block's P·V overwrites O.
      if (__any_sync(0xffffffffu, rescale && jj > 0)) {
        if (!mbar_wait_warp(bar_pv_done((jj - 1) & 1), ((jj - 1) >> 1) & 1u, wc, kSiteSmxPvDone))
          return false;
        tc_fence_after();
        const float a = (rescale && jj > 0) ? alpha : 1.f;
#pragma unroll
        for (int c0 = ch * kOCols; c0 < (ch + 1) * kOCols; c0 += 32) {
          uint32_t orow[32];
          tmem_ld_x32(tO + c0, orow);
#pragma unroll
          for (int c = 0; c < 32; ++c) orow[c] = __float_as_uint(__uint_as_float(orow[c]) * a);
          tmem_st_x32(tO + c0, orow);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p_full(buf));
      return true;
    };
    {
      // Blocks [ja, jb) of this CTA cross no mask boundary: every key visible at
      // every position of the tile (no ragged end, wholly inside both windows).
      int ja = 0, jb = nblocks;
      if (p.window_left >= 0) {  // key0 >= pos_max - window_left
        const int first = pos_max - p.window_left;
        if (first > 0) ja = max(ja, (first + kBN - 1) / kBN - it.lo);
      }
      jb = min(jb, Lk / kBN - it.lo);  // key0 + kBN <= Lk
      if (wr >= 0) {                   // key0 + kBN - 1 <= pos_min + wr
        const int last = pos_min + wr - (kBN - 1);
        jb = min(jb, last >= 0 ? last / kBN + 1 - it.lo : 0);
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
    if constexpr (kHalves == 2) {
      if (ok) {
        // the row sum over both halves (one more exchange round), same order in both
        float other = 0.f;
        ok = exchange(static_cast<uint32_t>(nblocks), l, other);
        l = (ch == 0) ? l + other : other + l;
      }
    }
    if (ok) {
      // ---- epilogue: O / l and the log-sum-exp of this row over this split; each
      // half of the row writes its half of the O columns
      const bool have = nblocks > 0;
      float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      if constexpr (PV16) inv_l *= exp2_int(-v16_exponent(p.vmax[it.b * p.Hkv + it.g]));
      const size_t row = (static_cast<size_t>(it.b) * p.Hq + h) * p.Lq + qi;  // LSE index
      const bool partial = p.splits > 1;
      const size_t nrows = static_cast<size_t>(p.B) * p.Hq * p.Lq;
#pragma unroll
      for (int c0 = ch * kOCols; c0 < (ch + 1) * kOCols; c0 += 32) {
        uint32_t orow[32];
        if (have) {
          tmem_ld_x32(tO + c0, orow);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) orow[c] = 0u;
        }
        if (!row_ok) continue;
        if (partial || OUT_F32) {
          float* dst = partial ? p.o_part + (static_cast<size_t>(it.split) * nrows + row) * D + c0
                               : static_cast<float*>(p.o) +
                                     ((static_cast<size_t>(it.b) * p.Lq + qi) * p.Hq + h) * D + c0;
          float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            d4[c >> 2] = make_float4(__uint_as_float(orow[c]) * inv_l,
                                     __uint_as_float(orow[c + 1]) * inv_l,
                                     __uint_as_float(orow[c + 2]) * inv_l,
                                     __uint_as_float(orow[c + 3]) * inv_l);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(
              static_cast<uint16_t*>(p.o) + ((static_cast<size_t>(it.b) * p.Lq + qi) * p.Hq + h) * D +
              c0);
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
      if (row_ok && ch == 0) {
        const float lse2 = (l > 0.f) ? m_ref + lg2_approx(l) : -INFINITY;  // base 2
        if (partial)
          p.lse_part[static_cast<size_t>(it.split) * nrows + row] = lse2;
        else if (p.lse != nullptr)
          p.lse[row] = (l > 0.f) ? lse2 * 0.69314718055994531f : -INFINITY;
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

// Combines the splits of each row: with L_s the partial log2-sum-exp of split s,
// L = log2 Σ_s 2^(L_s) and O = Σ_s 2^(L_s − L) · O_s. WPR warps per row, 8 warps per
// CTA: a decode call has a few rows and many splits, and one CTA per row (WPR = 8)
// makes that one round trip of loads; a square problem cut into splits has many rows
// and few splits, and one warp per row (WPR = 1) keeps the grid small. The warps of a
// row reduce the log-sum-exp over the splits, warp w of the row accumulates the
// weighted partial rows of splits w, w + WPR, ... (lane = D / 32 consecutive columns;
// up to 16 splits' loads in flight), and the partial sums meet in shared memory.
template <int D, bool BF16, bool OUT_F32, int WPR>
__global__ void __launch_bounds__(256) attn_kv_merge_kernel(const KvParams p) {
  static_assert(WPR == 1 || WPR == 8, "one warp or one CTA per row");
  // Launched as a programmatic dependent of the split kernel: its CTAs may start
  // while that kernel finishes; the partial results are read only after it is done.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int kCols = D / 32;
  constexpr int kWarps = 8;
  constexpr int kBatch = (WPR == 1) ? 8 : 16;  // splits per warp whose loads are in flight at once
  __shared__ float red[kWarps];
  __shared__ float part[kWarps][D];
  const size_t nrows = static_cast<size_t>(p.B) * p.Hq * p.Lq;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row = static_cast<size_t>(blockIdx.x) * (kWarps / WPR) + warp / WPR;
  const int sw = warp % WPR;  // this warp's index among the row's warps
  if constexpr (WPR == 1) {
    if (row >= nrows) return;  // no CTA-wide barrier in this mode
  }
  const int S = p.splits;
  // Reduction over the row's warps (a warp shuffle, then shared memory when WPR = 8).
  auto row_reduce = [&](float v, bool is_max) -> float {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float x = __shfl_xor_sync(0xffffffffu, v, o);
      v = is_max ? fmaxf(v, x) : v + x;
    }
    if constexpr (WPR > 1) {
      if (lane == 0) red[warp] = v;
      __syncthreads();
      v = red[0];
#pragma unroll
      for (int w = 1; w < WPR; ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
      __syncthreads();
    }
    return v;
  };
  float m = -INFINITY;
  for (int s = sw * 32 + lane; s < S; s += WPR * 32) m = fmaxf(m, p.lse_part[s * nrows + row]);
  m = row_reduce(m, true);
  float lse2 = -INFINITY;
  if (m != -INFINITY) {  // uniform over the row's warps
    float t = 0.f;
    for (int s = sw * 32 + lane; s < S; s += WPR * 32) t += exp2f(p.lse_part[s * nrows + row] - m);
    lse2 = m + log2f(row_reduce(t, false));
  }
  float acc[kCols];
#pragma unroll
  for (int c = 0; c < kCols; ++c) acc[c] = 0.f;
  if (lse2 != -INFINITY) {
    for (int s0 = sw; s0 < S; s0 += WPR * kBatch) {
      float wt[kBatch], v[kBatch][kCols];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int s = s0 + WPR * u;
        wt[u] = 0.f;
#pragma unroll
        for (int c = 0; c < kCols; ++c) v[u][c] = 0.f;
        if (s < S) {
          wt[u] = exp2f(p.lse_part[s * nrows + row] - lse2);  // 0 for an empty split
          const float* src = p.o_part + (s * nrows + row) * D + lane * kCols;
          if constexpr (kCols == 4) {
            const float4 x = *reinterpret_cast<const float4*>(src);
            v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
          } else {
            const float2 x = *reinterpret_cast<const float2*>(src);
            v[u][0] = x.x; v[u][1] = x.y;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (wt[u] != 0.f) {  // an empty split has weight 0 (and O_s = 0)
#pragma unroll
          for (int c = 0; c < kCols; ++c) acc[c] += wt[u] * v[u][c];
        }
    }
  }
  if constexpr (WPR > 1) {
#pragma unroll
    for (int c = 0; c < kCols; ++c) part[warp][lane * kCols + c] = acc[c];
    __syncthreads();
    if (warp != 0) return;
#pragma unroll
    for (int c = 0; c < kCols; ++c) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < WPR; ++w) t += part[w][lane * kCols + c];
      acc[c] = t;
    }
  }
  // the row's first warp writes O (lane = kCols consecutive columns) and the LSE
  const int qi = static_cast<int>(row % p.Lq);
  const int h = static_cast<int>((row / p.Lq) % p.Hq);
  const int b = static_cast<int>(row / (static_cast<size_t>(p.Lq) * p.Hq));
  const size_t o_off = ((static_cast<size_t>(b) * p.Lq + qi) * p.Hq + h) * D + lane * kCols;
  if constexpr (OUT_F32) {
    float* dst = static_cast<float*>(p.o) + o_off;
#pragma unroll
    for (int c = 0; c < kCols; ++c) dst[c] = acc[c];
  } else {
    uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.o) + o_off);
#pragma unroll
    for (int c = 0; c < kCols; c += 2) dst[c >> 1] = pack2(acc[c], acc[c + 1], BF16);
  }
  if (lane == 0 && p.lse != nullptr)
    p.lse[row] = (lse2 == -INFINITY) ? -INFINITY : lse2 * 0.69314718055994531f;
}

}  // namespace kv
}  // namespace ex19
