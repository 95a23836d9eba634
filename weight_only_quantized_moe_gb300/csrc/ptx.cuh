// ptx.cuh - inline-PTX wrappers for sm_103a: mbarriers, 1-D bulk TMA copies
// (cp.async.bulk) and the tcgen05 tensor-core / tensor-memory instructions.
//
// Every wait on an mbarrier here is bounded: it gives up after a time limit
// (measured with %globaltimer) or as soon as the CTA-wide abort flag is set,
// and reports which it was.  No wait in this library can spin forever.
#pragma once

#include <cstdint>

namespace qmoe {

// Limit for any single pipeline wait.  Real waits are micro-seconds; a wait
// that reaches this limit means the pipeline is broken and the kernel stops.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s
// Suspend-time hint of one try_wait: the thread wakes as soon as the phase
// completes; the hint only bounds one sleep, so the limit above stays checked.
constexpr uint32_t kSuspendHintNs = 1000000u;  // 1 ms

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: a kernel lets the next one in the stream start
// its prologue early (launch_dependents) and waits for the previous kernel's
// results to be complete and visible (wait) before it reads them.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// thread-block clusters (the GEMM's CTA-pair form)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of the cluster arrives; returns once all have (release / acquire
// at cluster scope, so barrier initialisation and shared-memory writes before it
// are visible to the other CTAs after it).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared::cluster address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_smem, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem), "r"(rank));
  return r;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

// Test for completion of the phase with the given parity.  The thread is
// suspended (it issues nothing) until the phase completes or the hinted time
// passes, so waiting warps do not take issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

// Arrive once on the barrier at shared::cluster address `remote_bar` (another
// CTA's, or this CTA's own through the cluster window).  Default semantics
// (release at CTA scope): the callers order their tensor-memory stores or loads
// with tcgen05.wait + tcgen05.fence::before_thread_sync and the waiter with
// tcgen05.fence::after_thread_sync, as for a local barrier; a release at cluster
// scope costs the arriving thread ~320 cycles (measured on GB300).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}

// Wait until the phase with the given parity has completed.  Returns false if
// the CTA abort flag was raised or the time limit passed (the caller then
// raises the abort flag itself and winds down).  Between polls the warp sleeps
// with exponential backoff up to `max_sleep_ns`, so waiting warps leave the
// issue slots to working ones; callers on the critical path pass a small cap.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int* abort_flag,
                                          uint32_t max_sleep_ns = 64) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t sleep_ns = 8;
  for (uint32_t it = 1;; ++it) {
    if (max_sleep_ns != 0) {
      __nanosleep(sleep_ns);
      sleep_ns = sleep_ns * 2 < max_sleep_ns ? sleep_ns * 2 : max_sleep_ns;
    }
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 7) == 0 && *abort_flag) return false;
    if ((it & 31) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Position in a ring of n pipeline slots plus the phase parity of the current lap.
struct Ring {
  int idx = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++idx == n) {
      idx = 0;
      phase ^= 1u;
    }
  }
  // Advance by r slots of a ring of n slots, n a multiple of r (a role that
  // takes every r-th stage).
  __device__ __forceinline__ void step(int r, int n) {
    idx += r;
    if (idx >= n) {
      idx -= n;
      phase ^= 1u;
    }
  }
};

// ---------------------------------------------------------------------------
// TMA (bulk async copies, completion counted on an mbarrier in bytes)
// ---------------------------------------------------------------------------
// Contiguous global -> shared copy; src, dst 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void tma_load_1d(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Shared-memory loads by shared-window address (the kernels align their dynamic
// shared memory through an integer, which leaves plain pointers generic).  The
// "memory" clobber keeps them after the barrier waits that publish the data.
__device__ __forceinline__ uint4 lds_u128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint2 lds_u64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

// Per-thread asynchronous 16-byte global -> shared copy (src, dst 16-byte aligned),
// completed by cp_async_wait_group (the thread's own copies; a __syncwarp after it
// makes them visible to the warp's other lanes).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed copy groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation tensor-core MMA
// ---------------------------------------------------------------------------
// Allocate `ncols` TMEM columns (power of two >= 32); one full warp executes it.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// The same for a CTA pair (cta_group::2): one warp in each CTA of the pair executes
// them with the same column count, and both CTAs receive the same TMEM address.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 1 in one lane of a converged warp, 0 in the others (the same lane for a full mask).
__device__ __forceinline__ uint32_t elect_one_sync() {
  uint32_t leader;
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, e;\n\t}"
      : "=r"(leader));
  return leader;
}

// The MMA and commit forms below are executed by a whole converged warp and issued
// by the lane whose `issue` is non-zero (elect_one_sync): their operands then stay
// warp-uniform, where a branch to one lane would have the compiler move every
// operand of every instruction from that lane into uniform registers.

// D[tmem] (+)= A[tmem] * B[smem]^T ; M = 128, N from idesc, K = 16 (16-bit types).
__device__ __forceinline__ void mma_ts_f16(uint32_t issue, uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(issue)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T with 2:4 structured sparsity in A: M = 128, N from idesc,
// K = 32 of the dense matrix per instruction (16-bit types); A holds the 16 kept values of each
// row (8 TMEM columns) and `meta_tmem` the 32-bit position words (one column, 8-column aligned
// like the A operand's steps).
__device__ __forceinline__ void mma_ts_sp_f16(uint32_t issue, uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t meta_tmem, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "setp.ne.b32 q, %6, 0;\n\t"
      "@q tcgen05.mma.sp.cta_group::1.kind::f16 [%0], [%1], %2, [%3], %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(meta_tmem), "r"(idesc), "r"(accumulate), "r"(issue)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by the issuing lane
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t issue, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred q;\n\t"
      "setp.ne.b32 q, %1, 0;\n\t"
      "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar),
      "r"(issue)
      : "memory");
}

// Pair MMA, issued from the even CTA of a CTA pair: D (+)= A * B^T with M = 256
// (rows 0-127 in the even CTA's TMEM lanes, 128-255 in the odd CTA's, A and D at
// the same TMEM address in both), N from idesc (each CTA's shared memory holds N/2
// rows of B at the same address), K = 16 (16-bit types).
__device__ __forceinline__ void mma_ts_f16_pair(uint32_t issue, uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(issue)
      : "memory");
}

// Arrive once on the barrier at this shared-memory offset in both CTAs of the pair
// when every tcgen05 operation issued so far by the issuing lane has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t issue, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred q;\n\t"
      "setp.ne.b32 q, %2, 0;\n\t"
      "@q tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(bar),
      "h"(static_cast<uint16_t>(0x3)), "r"(issue)
      : "memory");
}

// Instruction descriptor of kind::f16: D f32, A/B f16 or bf16, both K-major, M = 128.
__host__ __device__ __forceinline__ uint32_t make_idesc_m128(uint32_t n, bool bf16) {
  const uint32_t ab = bf16 ? 1u : 0u;
  return (1u << 4)             // D format: f32
         | (ab << 7)           // A format
         | (ab << 10)          // B format
         | ((n >> 3) << 17)    // N / 8
         | ((128u >> 4) << 24);  // M / 16
}

// The same with M = 256 (a CTA pair's MMA).
__host__ __device__ __forceinline__ uint32_t make_idesc_m256(uint32_t n, bool bf16) {
  const uint32_t ab = bf16 ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((n >> 3) << 17) | ((256u >> 4) << 24);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// `sbo` bytes apart (a multiple of 1024).  `saddr` may be offset by multiples
// of 32 bytes inside a 1024-byte aligned swizzle atom to step along K.
__device__ __forceinline__ uint64_t make_sdesc_k_sw128(uint32_t saddr, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused for swizzled K-major)
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;  // stride byte offset: next 8-row group
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                   // swizzle mode: 128 B
  return d;
}

// Warp-collective TMEM store: this warp's 32 lanes (lane quadrant from the
// address), 32 consecutive 32-bit columns per lane taken from v[OFF .. OFF+31].
template <int OFF, int N>
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&v)[N]) {
  static_assert(OFF + 32 <= N, "source range");
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[OFF + 0]), "r"(v[OFF + 1]), "r"(v[OFF + 2]), "r"(v[OFF + 3]), "r"(v[OFF + 4]), "r"(v[OFF + 5]),
      "r"(v[OFF + 6]), "r"(v[OFF + 7]), "r"(v[OFF + 8]), "r"(v[OFF + 9]), "r"(v[OFF + 10]), "r"(v[OFF + 11]),
      "r"(v[OFF + 12]), "r"(v[OFF + 13]), "r"(v[OFF + 14]), "r"(v[OFF + 15]), "r"(v[OFF + 16]), "r"(v[OFF + 17]),
      "r"(v[OFF + 18]), "r"(v[OFF + 19]), "r"(v[OFF + 20]), "r"(v[OFF + 21]), "r"(v[OFF + 22]), "r"(v[OFF + 23]),
      "r"(v[OFF + 24]), "r"(v[OFF + 25]), "r"(v[OFF + 26]), "r"(v[OFF + 27]), "r"(v[OFF + 28]), "r"(v[OFF + 29]),
      "r"(v[OFF + 30]), "r"(v[OFF + 31])
      : "memory");
}

// Warp-collective TMEM store: 16 consecutive 32-bit columns per lane.
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// Warp-collective TMEM store: one 32-bit column per lane.
__device__ __forceinline__ void tmem_st_32x32b_x1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Warp-collective TMEM load: 16 consecutive 32-bit columns per lane into v[OFF .. OFF+15].
template <int OFF = 0, int N = 16>
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&v)[N]) {
  static_assert(OFF + 16 <= N, "destination range");
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(v[OFF + 0]), "=r"(v[OFF + 1]), "=r"(v[OFF + 2]), "=r"(v[OFF + 3]), "=r"(v[OFF + 4]), "=r"(v[OFF + 5]),
        "=r"(v[OFF + 6]), "=r"(v[OFF + 7]), "=r"(v[OFF + 8]), "=r"(v[OFF + 9]), "=r"(v[OFF + 10]),
        "=r"(v[OFF + 11]), "=r"(v[OFF + 12]), "=r"(v[OFF + 13]), "=r"(v[OFF + 14]), "=r"(v[OFF + 15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace qmoe
