// Chunk scales from per-tile totals: scale = (sum of the chunk's tile
// totals, in tile order, from 0) / (real elements of the chunk), 0 for an
// all-padding chunk.  This is the last step of the fixed summation order
// of the mean |x| ("1-bit 梯度量化": mean(|g|) * sign(g)); running it as its
// own small kernel after the streaming kernels keeps those free of
// cross-CTA fences and counters.
//
// One warp per (row, chunk) sequence; rows are workers (compress) or the
// single server row.  The same ordered sum without the division finishes
// the error monitor's per-chunk sums of squares (k_monitor.cu).
#include "ob_internal.cuh"

namespace ob {
namespace {

template <bool MEAN>
__global__ void __launch_bounds__(kThreads)
    k_finalize_scales(const Geo G, const float* __restrict__ part, uint32_t rows, uint32_t g0,
                      uint32_t count, float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const uint32_t nseq = rows * count;
  for (uint32_t q = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); q < nseq;
       q += gridDim.x * (kThreads / 32)) {
    const uint32_t row = q / count;
    const uint32_t g = g0 + (q - row * count);
    const uint32_t kc = g % G.cpp;
    const uint32_t j = g / G.cpp;
    const bool last = kc == G.cpp - 1;
    const uint64_t clen = last ? G.Cl : G.C;
    const uint32_t ntc = last ? G.tpl : G.tpc;
    const uint64_t cstart = (uint64_t)j * G.P + (uint64_t)kc * G.C;
    const uint64_t real = G.n > cstart ? (G.n - cstart < clen ? G.n - cstart : clen) : 0;
    const float sum = ordered_sum(part + ((uint64_t)row * G.nc + g) * G.tpc, ntc, lane);
    if (lane == 0) scales[q] = MEAN ? mean_of(sum, real) : sum;
  }
}

}  // namespace

cudaError_t launch_finalize_scales_range(const Geo& G, const float* part, uint32_t rows,
                                         uint32_t g0, uint32_t count, float* scales, int sms,
                                         cudaStream_t s) {
  const uint64_t ctas = ((uint64_t)rows * count + kThreads / 32 - 1) / (kThreads / 32);
  k_finalize_scales<true><<<grid_for(k_finalize_scales<true>, sms, ctas), kThreads, 0, s>>>(
      G, part, rows, g0, count, scales);
  return cudaGetLastError();
}

cudaError_t launch_finalize_scales(const Geo& G, const float* part, uint32_t rows,
                                   float* scales, int sms, cudaStream_t s) {
  return launch_finalize_scales_range(G, part, rows, 0, G.nc, scales, sms, s);
}

cudaError_t launch_finalize_sums(const Geo& G, const float* part, uint32_t rows, float* sums,
                                 int sms, cudaStream_t s) {
  const uint64_t ctas = ((uint64_t)rows * G.nc + kThreads / 32 - 1) / (kThreads / 32);
  k_finalize_scales<false><<<grid_for(k_finalize_scales<false>, sms, ctas), kThreads, 0, s>>>(
      G, part, rows, 0, G.nc, sums);
  return cudaGetLastError();
}

}  // namespace ob
