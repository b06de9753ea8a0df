// Inline-PTX helpers for the bulk-copy pipelines: mbarriers in shared
// memory and cp.async.bulk (global -> shared, completion counted in bytes on
// an mbarrier).  Every wait is bounded: after kWaitCycles SM clocks it
// gives up, records an error code in the workspace and returns false, so a
// copy that never lands cannot hang the GPU.
#pragma once

#include <cstdint>

namespace ob {

// About one second at the GB300's 2 GHz maximum SM clock.
constexpr long long kWaitCycles = 2000000000LL;

// Error codes written to the workspace error word.
constexpr unsigned kErrWaitFull = 1;   // a consumer waited too long for a copy
constexpr unsigned kErrWaitEmpty = 2;  // the producer waited too long for a free stage
constexpr unsigned kErrDrain = 3;      // copies still in flight at exit

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Makes the initialised barriers visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits until the phase of `bar` with parity `parity` has completed, for at
// most `limit` SM clocks; on timeout records `code` in *err (if it holds no
// code yet) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err,
                                          unsigned code, long long limit = kWaitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) {
      atomicCAS(err, 0u, code);
      return false;
    }
  }
  return true;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory to this CTA's shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Asks the copy engine to bring `bytes` (multiple of 16; address 16-byte
// aligned) of global memory into L2.  A hint: nothing is returned to the
// SM and nothing waits for it.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Asynchronous 4- or 8-byte copy global -> this thread's view of shared
// memory (cp.async, no register holds the value); both addresses aligned to
// the size.  cp_async_wait_all() waits for this thread's copies; others see
// them only after a barrier.
__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Named barrier among the first `threads` threads of the CTA (id 1..15).
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also returns the OR of `v` over the participants, so
// every participant takes the same decision.
__device__ __forceinline__ bool named_sync_or(int id, int threads, bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)v), "r"(id), "r"(threads)
      : "memory");
  return out != 0;
}

}  // namespace ob
