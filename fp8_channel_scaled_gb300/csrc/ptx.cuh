// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA (bulk
// tensor copies), tcgen05 (tensor-memory MMA), cluster shared memory, and
// the bounded waits every kernel in this library uses.
//
// Every field layout below (shared-memory matrix descriptor, instruction
// descriptor, TMEM addresses) follows the PTX ISA description of the
// tcgen05 family; nothing here is taken from a compiled binary.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace fp8g {

// ----------------------------------------------------------------------------
// error codes a kernel can raise in the device error word (bit flags)
// ----------------------------------------------------------------------------
enum : unsigned {
  kErrWaitProducer = 1u << 0,   // producer gave up waiting for a free stage
  kErrWaitMma      = 1u << 1,   // MMA issuer gave up waiting for operands / accumulator
  kErrWaitEpilogue = 1u << 2,   // epilogue gave up waiting for an accumulator
  kErrWaitDrain    = 1u << 3,   // teardown gave up waiting for copies / MMAs in flight
  kErrWaitSelfTest = 1u << 4,   // the deliberate wait of the self-test kernel ran out
  kErrWaitPartial  = 1u << 5,   // a split tile's owner gave up waiting for a partial sum
};

// ----------------------------------------------------------------------------
// basic helpers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t warp_id() { return threadIdx.x >> 5; }
__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// ----------------------------------------------------------------------------
// mbarrier
// ----------------------------------------------------------------------------
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

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Per-CTA context of the bounded waits: where to report, how long to wait,
// and a shared-memory flag that makes every later wait of the CTA give up
// at once after the first one ran out.
struct WaitCtx {
  unsigned* err;             // device error word (global memory)
  volatile int* abort_flag;  // shared memory, 0 = keep going
  uint64_t budget_ns;        // longest single wait
};

// Slow path of mbar_wait_bounded (scalar arguments, so the call needs no
// stack frame).
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, unsigned* err,
                                                   volatile int* abort_flag, uint64_t budget_ns,
                                                   unsigned code) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > budget_ns) {
        *abort_flag = 1;
        atomicOr(err, code);
        return false;
      }
    }
  }
}

// Wait until the phase of `bar` with parity `parity` has completed.  Returns
// false (and records `code`) if it did not complete within the budget or if
// another wait of this CTA already gave up.  Never waits without limit.  The
// common case (phase already complete, or completing within one try_wait
// suspension) stays inline.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const WaitCtx& wc, unsigned code) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, wc.err, wc.abort_flag, wc.budget_ns, code);
}

// A wait used during teardown: ignores the abort flag (it must wait for work
// already in flight) but is still bounded.
static __device__ __noinline__ bool drain_wait(uint32_t bar, uint32_t parity, unsigned* err,
                                               uint64_t budget_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u && globaltimer_ns() - t0 > budget_ns) {
      atomicOr(err, kErrWaitDrain);
      return false;
    }
  }
}

// ----------------------------------------------------------------------------
// cross-CTA publication through global memory
// ----------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Wait until *flag == want (a value another CTA of the same grid publishes
// with st_release_u64).  Bounded like the mbarrier waits.
static __device__ __noinline__ bool flag_wait_bounded(const unsigned long long* flag,
                                                      unsigned long long want, unsigned* err,
                                                      volatile int* abort_flag,
                                                      uint64_t budget_ns) {
  if (ld_acquire_u64(flag) == want) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    __nanosleep(100);
    if (ld_acquire_u64(flag) == want) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > budget_ns) {
      *abort_flag = 1;
      atomicOr(err, kErrWaitPartial);
      return false;
    }
  }
}

// ----------------------------------------------------------------------------
// programmatic dependent launch
// ----------------------------------------------------------------------------
// Let the next kernel of the stream (launched with programmatic stream
// serialization) start its launch and prologue now; it still waits in
// griddep_wait() until this grid has completed.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the grids this kernel depends on have completed and their
// memory operations are visible.  A no-op when launched without programmatic
// stream serialization.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ----------------------------------------------------------------------------
// proxy fences
// ----------------------------------------------------------------------------
// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA engine, tensor cores).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's earlier generic-proxy global accesses (e.g. the acquire
// of a flag) before its later async-proxy global accesses (bulk copies).
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ----------------------------------------------------------------------------
// TMA
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Untiled bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to this CTA's shared memory, completing on `bar` as
// transaction bytes.
__device__ __forceinline__ void bulk_load_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// 2-D tiled load of one box into shared memory; completion is reported to
// the mbarrier as transaction bytes.  c0 is the innermost (byte) coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int32_t c0, int32_t c1,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Prefetch one box of a tiled tensor into L2: no shared-memory destination,
// no completion to wait for, no value returned to the thread.  L2 is the
// point of coherence for device memory, so a box prefetched before the
// preceding grid has finished writing it still reads as written by the
// later loads.  c0 (bytes) must be a multiple of 16.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}

// 3-D tiled load of one box into shared memory with an L2 cache hint.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int32_t c0, int32_t c1,
                                                 int32_t c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

// L2 prefetch of one box of a 3-D tiled tensor (as tma_prefetch_l2_2d).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int32_t c0, int32_t c1,
                                                   int32_t c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// 2-D tiled store of one box from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                             int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed store groups still read shared memory.
template <int N>
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// ----------------------------------------------------------------------------
// tcgen05: tensor memory and MMA
// ----------------------------------------------------------------------------
// Allocate ncols TMEM columns (power of two, >= 32); the TMEM address is
// written to shared memory.  Whole warp.
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

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, E4M3 x E4M3 -> F32, one thread.
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor for kind::f8f6f4: D = F32, A = B = E4M3, both
// K-major, no negation, dense.  Fields: [4,6) D format (1 = F32),
// [7,10) A format (0 = E4M3), [10,13) B format (0 = E4M3), bit 15/16
// major-ness (0 = K), [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t m, uint32_t n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms
// stacked along M/N.  Fields: [0,14) start address >> 4, [16,30) leading
// byte offset >> 4 (unused for a swizzled K-major tile whose MMA K-slice
// stays inside one 128-byte row), [32,46) stride byte offset >> 4 = 1024
// between 8-row groups, [46,48) descriptor version 1, [61,64) layout
// 2 = 128-byte swizzle.  The tile base must be 1024-byte aligned; advancing
// along K inside the row is done by adding bytes>>4 to the start address.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(16u >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// 32 TMEM lanes x 32 consecutive 32-bit columns -> 32 registers per thread
// (thread t of the warp receives lane base+t).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ----------------------------------------------------------------------------
// tcgen05 on a CTA pair (cta_group::2): the even CTA of a 2-CTA cluster issues
// MMAs whose A rows and B rows are split between the two CTAs' shared memory
// (same offsets) and whose accumulator rows live in both CTAs' TMEM.
// ----------------------------------------------------------------------------
// Collective: one warp in each CTA of the pair executes it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

// Collective: one warp in each CTA of the pair executes it.
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// One pipeline stage of the CTA-pair MMA issuer in a single asm block:
//   - test (without blocking) whether the next stage's full barrier
//     `next_full` has completed phase `next_parity`;
//   - issue 4 MMAs (K = 32 each) over the stage's first 128-byte K block
//     (accumulating if `accumulate`, else overwriting D for the first one),
//     and 4 more over its second K block if `two_kb`;
//   - commit the stage to the mbarrier `empty` in the CTAs of `cta_mask`;
//   - return the test's result.
// The barrier test is issued first and its result read last, so its latency
// overlaps the MMA issue instead of adding to it.  a_step / b_step: offset
// of the second K block in descriptor units (bytes / 16).
__device__ __forceinline__ bool tc_mma_stage_pair(uint32_t d_tmem, uint64_t a_desc,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate, uint32_t two_kb,
                                                  uint64_t a_step, uint64_t b_step,
                                                  uint32_t empty, uint16_t cta_mask,
                                                  uint32_t next_full, uint32_t next_parity) {
  uint32_t ready;
  asm volatile(
      "{\n\t"
      ".reg .pred pr, pa, ph, pt;\n\t"
      ".reg .b64 a1, b1;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 pr, [%10], %11;\n\t"
      "setp.ne.b32 pa, %5, 0;\n\t"
      "setp.ne.b32 ph, %6, 0;\n\t"
      "setp.eq.b32 pt, 0, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%1], %2, %3, %4, pa;\n\t"
      "add.s64 a1, %2, 2;\n\t"
      "add.s64 b1, %3, 2;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%1], a1, b1, %4, pt;\n\t"
      "add.s64 a1, %2, 4;\n\t"
      "add.s64 b1, %3, 4;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%1], a1, b1, %4, pt;\n\t"
      "add.s64 a1, %2, 6;\n\t"
      "add.s64 b1, %3, 6;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%1], a1, b1, %4, pt;\n\t"
      "add.s64 a1, %2, %7;\n\t"
      "add.s64 b1, %3, %8;\n\t"
      "@ph tcgen05.mma.cta_group::2.kind::f8f6f4 [%1], a1, b1, %4, pt;\n\t"
      "add.s64 a1, a1, 2;\n\t"
      "add.s64 b1, b1, 2;\n\t"
      "@ph tcgen05.mma.cta_group::2.kind::f8f6f4 [%1], a1, b1, %4, pt;\n\t"
      "add.s64 a1, a1, 2;\n\t"
      "add.s64 b1, b1, 2;\n\t"
      "@ph tcgen05.mma.cta_group::2.kind::f8f6f4 [%1], a1, b1, %4, pt;\n\t"
      "add.s64 a1, a1, 2;\n\t"
      "add.s64 b1, b1, 2;\n\t"
      "@ph tcgen05.mma.cta_group::2.kind::f8f6f4 [%1], a1, b1, %4, pt;\n\t"
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%9], %12;\n\t"
      "selp.b32 %0, 1, 0, pr;\n\t"
      "}\n"
      : "=r"(ready)
      : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(two_kb),
        "l"(a_step), "l"(b_step), "r"(empty), "r"(next_full), "r"(next_parity), "h"(cta_mask)
      : "memory");
  return ready != 0;
}

// Arrive once on the mbarrier at this shared-memory offset in every CTA of
// `cta_mask` when all pair MMAs this thread issued have completed.
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier that may live in the peer CTA (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}

// 3-D variant of tma_load_2d_pair.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1,
                                                 int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Arrive on an mbarrier given by its cluster address (possibly another CTA's)
// with the default semantics, release at CTA scope: the arrive orders nothing
// of this thread's memory for the peer CTA.  It serves as the signal that this
// warp's tensor-memory reads are over, and those are complete before it
// (tcgen05.wait::ld, then tcgen05.fence::before_thread_sync).  A release at
// cluster scope would first wait until every earlier write of the thread is
// visible to the whole cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// ----------------------------------------------------------------------------
// clusters and distributed shared memory
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of cluster_sync_all, for threads that arrive now and wait
// later (each thread must wait before it arrives again).
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ float4 ld_dsmem_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ----------------------------------------------------------------------------
// plain memory helpers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void sts_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void sts_f32(uint32_t addr, float a) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(a) : "memory");
}

// Pack two floats into a bf16x2 word, round to nearest even; lo goes to the
// lower address.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace fp8g
