// Test-only kernels for the bounded mbarrier wait the pipelined kernels use
// (csrc/ptx.cuh): a wait on a barrier that nothing completes must give up
// after its limit, record its code in the error word and let the kernel
// return; a wait on a completed phase must succeed at once.  Built by
// tests/test_gpu_waits.py with nvcc into a temporary shared library.
#include <cstdint>

#include "ptx.cuh"

namespace {

__global__ void k_wait_selftest(unsigned* err, long long limit, int arrive_first,
                                int* result, long long* cycles) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ob::mbar_init(&bar, 1);
    ob::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (arrive_first) ob::mbar_arrive(&bar);  // completes phase 0
    const long long t0 = clock64();
    const bool ok = ob::mbar_wait(&bar, 0, err, ob::kErrWaitFull, limit);
    cycles[0] = clock64() - t0;
    result[0] = ok ? 1 : 0;
  }
}

}  // namespace

extern "C" int wait_selftest(unsigned* err, long long limit, int arrive_first, int* result,
                             long long* cycles) {
  k_wait_selftest<<<1, 32>>>(err, limit, arrive_first, result, cycles);
  if (cudaGetLastError() != cudaSuccess) return 1;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 2;
}
