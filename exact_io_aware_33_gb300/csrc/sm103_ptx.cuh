// Inline-PTX building blocks for sm_103a: mbarriers, TMA tensor loads,
// tcgen05 (TMEM allocation, MMA, commit, TMEM loads/stores) and the shared
// memory matrix descriptors the tensor core reads operands through.
//
// Every wait in this file is bounded: it gives up after a fixed wall-clock
// budget (read from %globaltimer) or as soon as another role of the CTA has
// raised the CTA's abort flag, and reports that to the caller, which then
// winds down instead of spinning forever.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// ---------------------------------------------------------------- status
enum : int {
  kStatusOk = 0,
  kStatusTimeout = 1,       // a bounded wait ran out
};

// Wall-clock budget of a single wait, in nanoseconds (about one second; a
// test-only build of the timeout path sets a few milliseconds).
#ifdef FA_WAIT_BUDGET_NS
constexpr unsigned long long kWaitBudgetNs = FA_WAIT_BUDGET_NS;
#else
constexpr unsigned long long kWaitBudgetNs = 1000ull * 1000ull * 1000ull;
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- launch overlap
// Every kernel of this library is launched with programmatic stream
// serialization allowed, so its CTAs may start while the kernel before it on
// the stream is still running. Each kernel calls grid_dep_wait() before its
// first global-memory access (only shared-memory set-up, tensor-memory
// allocation and tensor-map prefetches come earlier): it returns once that
// kernel has completed and its writes are visible (at once when there is no
// such kernel). grid_dep_launch() then lets the next kernel's CTAs start;
// because it follows the wait, a kernel never overlaps the one two places
// before it.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }
__device__ __forceinline__ uint32_t warp_id() { return threadIdx.x >> 5; }

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One arrival for the whole warp, from lane 0 once every lane has reached
// this point: the warp barrier orders each lane's earlier shared-memory and
// (waited-for) tensor-memory writes before lane 0's releasing arrive. A
// barrier fed this way counts warps, not threads. Thirty-two lanes arriving
// one by one on the same barrier word are serialised by the shared-memory
// pipe, which the tensor core also reads its operands through.
// All 32 lanes must call it together.
__device__ __forceinline__ void mbar_arrive_warp(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31u) == 0) mbar_arrive(bar);
}

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

// Wait until the phase of parity `parity` of barrier `bar` has completed.
// Returns false (and raises *abort) when the wait budget runs out, or
// returns false at once when *abort is already raised by another role.
// With abort == nullptr the wait ignores other roles and only the budget
// ends it (used to drain copies and MMAs in flight before the CTA exits).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_test(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (global_ns() - t0 > kWaitBudgetNs) {
      if (abort != nullptr) *abort = 1;
      return false;
    }
  }
}

// try_wait with a suspend-time hint: the thread sleeps in hardware until the
// phase completes or about kSuspendHintNs pass. Waking takes longer than a
// poll notices the phase, so this suits waits off the critical path, where
// polling would only take issue slots from the warps doing the work.
constexpr uint32_t kSuspendHintNs = 1000000u;
__device__ __forceinline__ bool mbar_try_suspend(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// mbar_wait with sleeping instead of polling; same budget and abort rules.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_suspend(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_suspend(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (global_ns() - t0 > kWaitBudgetNs) {
      if (abort != nullptr) *abort = 1;
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box into shared memory; completion is signalled on
// `bar` as transaction bytes. Coordinates are element indices, innermost
// first; x (c0) must be a multiple of 8 for 16-bit data (16-byte rule).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// L2 policy for data read once: its lines are the first to be evicted, so it
// does not push out lines that are read again.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// tma_load_3d with an L2 cache policy (policy_evict_first) for the loaded lines.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int c0, int c1, int c2, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(pol)
      : "memory");
}

// 3-D tiled store of one box from shared memory (the layout the map's swizzle
// implies) to global memory, in the thread's current bulk group. Rows past
// the tensor's extent are not written. The source may be rewritten after
// bulk_wait_read<0>() following the group's commit.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// 1-D bulk copy global -> shared, completion as transaction bytes on `bar`.
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Bulk reduction shared -> global: adds `bytes` bytes of fp32 values at
// `src` element-wise into `dst` (both 16-byte aligned, size a multiple of
// 16). The copy engine reads the source asynchronously: the source may only
// be rewritten after bulk_wait_read<0>() (or <n> with n groups allowed to
// stay in flight) following the commit of this copy's group.
__device__ __forceinline__ void bulk_reduce_add_f32(float* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                   reinterpret_cast<uint64_t>(dst)),
               "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed bulk groups still read their shared source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until at most N committed bulk groups are still incomplete (their
// global writes included).
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Fire-and-forget 16-byte add into global memory (no value returned).
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// ---------------------------------------------------------------- fences
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- registers
// Per-warpgroup register budget (all four warps of the warpgroup execute
// it). The increases of a CTA are served from what its decreases free, so
// the new budgets, summed over warpgroups, must fit in the registers the
// CTA was launched with.
template <uint32_t R>
__device__ __forceinline__ void regs_increase() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <uint32_t R>
__device__ __forceinline__ void regs_decrease() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}

// ---------------------------------------------------------------- TMEM
// Allocation is warp-wide; the TMEM address lands in shared memory at `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
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

// TMEM address of (lane, column).
__device__ __forceinline__ uint32_t tmem_at(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

#define FA_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                 "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define FA_W8(i) "r"(r[i + 0]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                 "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
#define FA_RW8(i) "+r"(r[i + 0]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), \
                  "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives
// lane (base lane + t), columns col .. col+31. The values are not usable
// before tmem_ld_wait(r) (which ties them to the wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24)
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : FA_R8(0), FA_R8(8)
      : "r"(taddr)
      : "memory");
}

// Wait for this thread's outstanding TMEM loads; the register operands make
// every later use of the loaded values depend on the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : FA_RW8(0), FA_RW8(8), FA_RW8(16), FA_RW8(24)
               :
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : FA_RW8(0), FA_RW8(8) : : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      FA_W8(0), FA_W8(8), FA_W8(16), FA_W8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      FA_W8(0), FA_W8(8)
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- MMA
// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A and B and an
// fp32 accumulator. a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, bool a_mn, bool b_mn) {
  return (1u << 4)                      // D format: f32
         | (1u << 7)                    // A format: bf16
         | (1u << 10)                   // B format: bf16
         | ((a_mn ? 1u : 0u) << 15)     // A major
         | ((b_mn ? 1u : 0u) << 16)     // B major
         | ((N >> 3) << 17)             // N / 8
         | ((M >> 4) << 24);            // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle. `addr` is the shared
// address of the (1024-byte aligned) swizzle atom the operand starts in,
// possibly advanced along K inside the atom; lbo / sbo are byte offsets.
//   K-major  : sbo = distance between 8-row groups; lbo unused.
//   MN-major : lbo = distance between 64-element groups along M/N,
//              sbo = distance between 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;                      // descriptor version for tcgen05
  d |= 2ull << 61;                      // swizzle mode: 128 bytes
  return d;
}

// D[tmem] (+)= A[smem] * B[smem]^T   (one instruction, K = 16 for bf16)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Warp-wide forms of the three calls above, for an issuing warp whose 32
// lanes run the issue loop together: one elected lane (the lowest, lane 0
// in a converged warp) issues, so every commit tracks the MMAs before it.
// With the whole warp converged the descriptors and TMEM addresses stay
// warp-uniform, and a TS MMA (A in TMEM, N = 64) issues in ~32 cycles
// instead of ~45 from a lone lane under a branch. All 32 lanes must call
// them together.
__device__ __forceinline__ void mma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit_w(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// mbar_wait by all 32 lanes of a warp, with one verdict for all of them (a
// lane that gave up makes the whole warp give up), so the warp stays
// converged for the elected issue above.
__device__ __forceinline__ bool mbar_wait_w(uint32_t bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

// mbar_wait_sleep by all 32 lanes of a warp, with one verdict for all.
__device__ __forceinline__ bool mbar_wait_sleep_w(uint32_t bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait_sleep(bar, parity, abort));
}

// ---------------------------------------------------------------- math
// 3-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of 32 consecutive values.
__device__ __forceinline__ float max32(const float* x) {
  float m = x[0];
#pragma unroll
  for (int i = 1; i < 31; i += 2) m = max3(m, x[i], x[i + 1]);
  return fmaxf(m, x[31]);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two floats to a bf16 pair (round to nearest even): lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------- dropout keep bytes
// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC 2011): ten rounds, each forming the 64-bit products
// of counter words 0 and 2 with two fixed odd multipliers and replacing the
// counter by (hi2 ^ c1 ^ k0, lo2, hi0 ^ c3 ^ k1, lo0); the key grows by two
// Weyl increments before every round after the first.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = c.x * 0xD2511F53u, hi0 = __umulhi(c.x, 0xD2511F53u);
    const uint32_t lo1 = c.z * 0xCD9E8D57u, hi1 = __umulhi(c.z, 0xCD9E8D57u);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// Exchange with lane ^ mask: send `if_set` when bit is 1, else `if_clear`.
__device__ __forceinline__ uint32_t shfl_xor_sel(uint32_t bit, uint32_t if_set, uint32_t if_clear, int mask) {
  return __shfl_xor_sync(0xffffffffu, bit ? if_set : if_clear, mask);
}

// Dropout keep bytes. One generator call covers a 4 x 4 block of (query,
// key) pairs: counter (key >> 2, query >> 2, batch-head, offset), output
// word (query & 3), byte (key & 3). Lanes 4m..4m+3 of a warp own four
// consecutive rows of one kind (queries in the forward, keys in the
// backward, lane & 3 = row & 3) and need the same 16 columns of the other
// kind: lane r makes the call for column group r and the four words are
// exchanged among the quad in four shuffles. On return out[g] holds this
// lane's four bytes of column group g (byte c = column 4g + c).
//   row_major = true:  calls are indexed (column group, row group): the
//                      forward (rows = queries, columns = keys)
//   row_major = false: (row group, column group) and each word is
//                      transposed first: the backward (rows = keys,
//                      columns = queries)
template <bool kRowsAreQueries>
__device__ __forceinline__ void keep_bytes_quad(uint32_t row_group, uint32_t col_group0, uint32_t bh,
                                                uint32_t offset, uint32_t seed_lo, uint32_t seed_hi,
                                                uint32_t (&out)[4]) {
  const uint32_t r = threadIdx.x & 3u;
  const uint32_t col_group = col_group0 + r;
  const uint4 w = kRowsAreQueries
                      ? philox4x32_10(make_uint4(col_group, row_group, bh, offset), seed_lo, seed_hi)
                      : philox4x32_10(make_uint4(row_group, col_group, bh, offset), seed_lo, seed_hi);
  uint32_t t0, t1, t2, t3;  // t_j: what lane j of the quad needs from this call
  if constexpr (kRowsAreQueries) {
    t0 = w.x; t1 = w.y; t2 = w.z; t3 = w.w;  // word q: query q's four keys
  } else {
    // key k of the block needs byte k of each query word: 4 x 4 byte transpose
    const uint32_t lo01 = __byte_perm(w.x, w.y, 0x5140), hi01 = __byte_perm(w.x, w.y, 0x7362);
    const uint32_t lo23 = __byte_perm(w.z, w.w, 0x5140), hi23 = __byte_perm(w.z, w.w, 0x7362);
    t0 = __byte_perm(lo01, lo23, 0x5410);
    t1 = __byte_perm(lo01, lo23, 0x7632);
    t2 = __byte_perm(hi01, hi23, 0x5410);
    t3 = __byte_perm(hi01, hi23, 0x7632);
  }
  // 4 x 4 transpose of words across the quad: lane j needs word j of every
  // lane's call. Two butterfly exchanges (lane bit 0, then bit 1), each
  // sending the two words whose index differs from the lane in that bit.
  const uint32_t b0 = r & 1u, b1 = (r >> 1) & 1u;
  const uint32_t s0 = shfl_xor_sel(b0, t0, t1, 1), s1 = shfl_xor_sel(b0, t2, t3, 1);
  const uint32_t n0 = b0 ? s0 : t0, n1 = b0 ? t1 : s0, n2 = b0 ? s1 : t2, n3 = b0 ? t3 : s1;
  const uint32_t u0 = shfl_xor_sel(b1, n0, n2, 2), u1 = shfl_xor_sel(b1, n1, n3, 2);
  // out[g]: this lane's part of lane g's call, i.e. of column group g
  out[0] = b1 ? u0 : n0;
  out[1] = b1 ? u1 : n1;
  out[2] = b1 ? n2 : u0;
  out[3] = b1 ? n3 : u1;
}

// Dropout keep test on the four bytes of a word at once (an element is kept
// when its byte is >= t, t in [0, 255]). Per byte b, (b | 0x80) - t' cannot
// borrow from the next byte for t' <= 128, and its top bit says whether the
// low seven bits of b reach t'. For t <= 128 a byte is kept when its top bit
// is set or the low bits reach t (t' = t); for t > 128 only when its top
// bit is set and the low bits reach t - 128 (t' = t - 128).
struct KeepTest {
  uint32_t t4;    // t' in every byte
  uint32_t high;  // all ones when t > 128
};
__device__ __forceinline__ KeepTest keep_test(uint32_t t) {
  const bool hi = t > 128u;
  return KeepTest{(hi ? t - 128u : t) * 0x01010101u, hi ? 0xffffffffu : 0u};
}
// 0x80 in each byte of w that is kept, 0 in each byte that is dropped.
__device__ __forceinline__ uint32_t keep_bits4(uint32_t w, KeepTest k) {
  const uint32_t x = (w | 0x80808080u) - k.t4;
  return (((w & x) & k.high) | ((w | x) & ~k.high)) & 0x80808080u;
}
// prmt with sign replication: each selector nibble 8 + i fills its result
// byte with the top bit of byte i of a, so keep bits become byte masks
// (0x9988: bytes 0, 1 -> the low and high halves of a bf16 pair; 0x8888:
// byte 0 -> a whole 32-bit word).
template <uint32_t kSel>
__device__ __forceinline__ uint32_t sign_bytes(uint32_t a) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %1, %2;" : "=r"(d) : "r"(a), "n"(kSel));
  return d;
}

}  // namespace fa
