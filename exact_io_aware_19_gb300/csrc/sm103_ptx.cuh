// sm103_ptx.cuh — inline-PTX building blocks for the sm_103a attention kernel:
// mbarriers with bounded waits, TMA tile loads, TMEM allocation, tcgen05 MMA /
// commit / fences, and the shared-memory and instruction descriptors of tcgen05.
//
// Descriptor encodings follow the PTX ISA (tcgen05 "shared memory descriptor" and
// "instruction descriptor" for .kind::f16); the field positions are the ones
// written in each encoder below.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace ex19 {

// ---------------------------------------------------------------- status words
// The device status word (in the caller's workspace): [0] = attn_status_t code of
// the first error, [1] = where it happened (role << 16 | site), [2] = CTA, [3] = unit.
enum : uint32_t { kStatusInvalidArg = 1, kStatusWorkspace = 3, kStatusTimeout = 5 };  // attn_status_t codes

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------- mbarriers
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// One non-blocking probe: true once the phase with parity `parity` has completed.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe (never suspends): used instead of the potentially blocking
// try_wait when the wait limit is shorter than kMaxSuspendNs.
__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Probe with a suspend-time hint: a thread whose phase is not complete sleeps in
// hardware until the phase completes or `hint_ns` passes, instead of spinning and
// taking issue slots from the warps that do the work.
__device__ __forceinline__ bool mbar_test_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Longest single sleep of a waiting thread (1 ms): also the worst-case time a role
// takes to notice that another role of its CTA has aborted.
constexpr uint64_t kMaxSuspendNs = 1000000ull;
// Waits that drain copies and MMAs already issued (after an abort) run for at least
// this long (1 s), whatever the configured limit: those operations always complete,
// and the CTA must not free its shared memory or TMEM while they are in flight.
constexpr uint64_t kDrainFloorNs = 1000000000ull;

// Shared control block of one CTA for bounded waits.
struct WaitCtl {
  volatile uint32_t* abort_flag;  // shared memory: set once any role gives up
  uint32_t* status;               // global status word (may be null)
  uint64_t limit_ns;              // per-wait limit
  uint32_t unit;                  // current work unit, for the report
  uint32_t hint_ns;               // sleep hint of one poll: min(limit, kMaxSuspendNs)
  uint64_t drain_ns;              // limit of drain waits: max(limit, kDrainFloorNs)
  // Limits shorter than kMaxSuspendNs: every probe is non-blocking, so a wait runs
  // out as soon as it has waited for longer than the limit. (A potentially blocking
  // try_wait may sleep in hardware until its phase completes, for a time the
  // hardware chooses, before the limit is ever looked at.)
  bool poll_only;
  __device__ __forceinline__ void set_limit(uint64_t ns) {
    limit_ns = ns;
    hint_ns = static_cast<uint32_t>(ns < kMaxSuspendNs ? ns : kMaxSuspendNs);
    drain_ns = ns > kDrainFloorNs ? ns : kDrainFloorNs;
    poll_only = ns < kMaxSuspendNs;
  }
};

__device__ __forceinline__ void record_error(const WaitCtl& c, uint32_t code, uint32_t where) {
  *c.abort_flag = 1u;
  if (c.status != nullptr) {
    if (atomicCAS(c.status, 0u, code) == 0u) {
      c.status[1] = where;
      c.status[2] = blockIdx.x;
      c.status[3] = c.unit;
      __threadfence();
    }
  }
}

// Slow path of a bounded wait: polls until phase `parity` of `bar` completes, the
// limit runs out (recording a timeout) or, when `honor_abort`, another role of
// the CTA has aborted. Returns true only when the phase completed. The sleep hint
// never exceeds the limit, so a short limit times out as soon as a wait has to wait.
// Drain waits (`honor_abort` false) use at least kDrainFloorNs.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                            uint32_t where, bool honor_abort) {
  const uint64_t t0 = globaltimer_ns();
  const uint64_t limit = honor_abort ? c.limit_ns : c.drain_ns;
  while (true) {
    if (c.poll_only ? mbar_poll(bar, parity) : mbar_test_sleep(bar, parity, c.hint_ns)) return true;
    if (honor_abort && *c.abort_flag) return false;
    if (globaltimer_ns() - t0 >= limit) {
      record_error(c, kStatusTimeout, where);
      return false;
    }
  }
}

// Waits for phase `parity` of `bar`; false (never an endless wait) on timeout or abort.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                                  uint32_t where) {
  if (c.poll_only ? mbar_poll(bar, parity) : mbar_test(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, c, where, true);
}

// Same, but keeps waiting after an abort: used to let in-flight copies and MMAs
// finish before the CTA releases its TMEM and exits.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                                uint32_t where) {
  if (c.poll_only ? mbar_poll(bar, parity) : mbar_test(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, c, where, false);
}

// Whole-warp wait: every lane polls, then the warp agrees (all lanes must see the
// phase complete), so the .sync.aligned tcgen05 instructions that follow are
// always executed by the full warp or by none of it.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                               uint32_t where) {
  const bool ok = mbar_wait_bounded(bar, parity, c, where);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------------- TMA
// 4-D tiled bulk-tensor load into shared memory, completing on `bar` with the
// copied byte count. Coordinates are element indices, innermost first; the
// innermost coordinate times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

// 2-D tiled bulk-tensor load (same rules as tma_load_4d).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// One float from shared memory.
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Barrier `id` (1..15) over the first `count` threads of the CTA (a multiple of 32).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}


__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Brings the 4-D box at (c0, c1, c2, c3) of `map` into L2 (a hint: nothing is written
// to shared memory and no barrier is signalled; out-of-range parts are skipped).
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* map, int c0, int c1, int c2,
                                                   int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

// ------------------------------------------------------------------------ TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 16 zero bytes to shared memory (generic proxy).
__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tcgen05.mma operand reads) that is ordered after it.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05 MMA
// D[tmem] (+)= A · B[smem desc], A from a shared-memory descriptor (SS) or TMEM (TS).
// Warp-collective forms: the whole warp calls them convergently (so operands can
// sit in uniform registers) and one lane, picked by elect.sync, issues.
__device__ __forceinline__ void mma_ss_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (+)= A · B for float8 e4m3 A and B, both in shared memory (.kind::f8f6f4,
// K = 32 per instruction); issued by one lane picked by elect.sync. The
// instruction descriptor has the .kind::f16 layout with format 0 (e4m3) for both.
__device__ __forceinline__ void mma_ss_f8_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with A (e4m3) in TMEM: each 32-bit column holds 4 consecutive K values of
// its lane's row, so one MMA of K = 32 reads 8 columns.
__device__ __forceinline__ void mma_ts_f8_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16-bit A in TMEM (two K values per 32-bit column: one MMA of K = 16 reads 8 columns).
__device__ __forceinline__ void mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation the issuing lane has issued so far
// is done (one lane, picked by elect.sync, commits).
__device__ __forceinline__ void mma_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor, 128-byte swizzle:
//   bits  0-13 start address >> 4      bits 16-29 leading-dimension byte offset >> 4
//   bits 32-45 stride byte offset >> 4 bits 46-47 descriptor version (1)
//   bits 49-51 base offset (0: atoms are 1024-byte aligned)
//   bits 61-63 layout (2 = 128-byte swizzle)
// K-major operand: rows of 128 bytes, 8-row atoms `sbo` apart (lbo unused).
// MN-major operand: 64-element row segments, `lbo` = distance between 64-wide
// segments along MN, `sbo` = distance between groups of 8 rows along K.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// The same with another swizzle layout (bits 61-63): 2 = 128-byte, 4 = 64-byte.
// K-major tiles with 64-byte rows (64 float8 elements) use the 64-byte swizzle,
// whose 8-row atom is 512 bytes (sbo).
__device__ __forceinline__ uint64_t sdesc_swizzled(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                                   uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}

// Instruction descriptor, .kind::f16, dense, fp32 accumulator:
//   bits 4-5 D format (1 = f32)   bits 7-9 A format, 10-12 B format (0 = f16, 1 = bf16)
//   bit 15 A major (0 = K)        bit 16 B major (0 = K, 1 = MN)
//   bits 17-22 N >> 3             bits 24-28 M >> 4
__host__ __device__ constexpr uint32_t idesc_f16_f32acc(bool bf16, int M, int N, bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// The same with either operand's major-ness: A MN-major (bit 15) reads A[m][k] with m
// contiguous (64-element segments `lbo` apart, 8-element groups of k `sbo` apart).
__host__ __device__ constexpr uint32_t idesc_f16_f32acc_ab(bool bf16, int M, int N, bool a_mn_major,
                                                         bool b_mn_major) {
  return idesc_f16_f32acc(bf16, M, N, b_mn_major) | ((a_mn_major ? 1u : 0u) << 15);
}

// -------------------------------------------------------------------- arithmetic
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three-input maximum (one instruction on sm_100+).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two exponentials in one MUFU operation: (2^a, 2^b) for a packed pair of fp16
// arguments, result packed as fp16 (low half = first element).
__device__ __forceinline__ uint32_t ex2_f16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace ex19
