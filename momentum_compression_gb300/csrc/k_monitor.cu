// The quantisation-error monitor of the 1-bit path (gradient quantization
// tutorial, "监控与诊断": watch the norm of the quantisation error; "1bit
// Adam" write-up §7: check that the error term stays bounded): per chunk,
// the sum of the squared true errors of every worker and of the server.
//
// The errors are held in the deferred form, so each one is decoded first,
// e' = x - (bit ? scale : -scale), exactly as the next compression would.
// Each CTA takes whole 4096-element tiles; for every row (the W workers,
// then the server) lane p adds the squares of elements 1024*i + 4*p + c
// (i, c = 0..3, real elements only) from a 128-bit load, the warps are
// reduced by butterflies and the 8 warp totals by the pairwise tree -- the
// fixed order of every scale here -- and the tile total goes to the
// workspace.  The ordered sum of a chunk's tile totals is the finalize
// kernel's, without the division.
#include "ob_internal.cuh"

namespace ob {
namespace {

__global__ void __launch_bounds__(kThreads) k_error_norm(const MaterializeArgs A, Workspace ws) {
  const Geo& G = A.geo;
  const int p = threadIdx.x, lane = p & 31, warp = p >> 5;
  __shared__ float wsum[kThreads / 32];
  for (uint32_t T = blockIdx.x; T < G.n_tiles; T += gridDim.x) {
    const Tile tl = decode_tile(G, T);
    for (uint32_t r = 0; r <= G.W; ++r) {
      // r < W: worker r's error; r == W: the server's
      const float* e = r < G.W ? A.e[r] : A.e_s;
      const uint32_t* bw = r < G.W ? A.bits + (uint64_t)r * G.words : A.sbits;
      const float sc = r < G.W ? __ldcg(A.scales + (uint64_t)r * G.nc + tl.g)
                               : __ldcg(A.sscales + tl.g);
      float acc = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t off = 1024u * i + 4u * p;
        const uint64_t k0 = tl.start + off;
        if (off >= tl.len || k0 >= G.n) continue;
        const float4 xv = __ldcs(reinterpret_cast<const float4*>(e + k0));
        const uint32_t wd = __ldcs(bw + (k0 >> 5)) >> (k0 & 31);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (k0 + c >= G.n) continue;
          const float so = ((wd >> c) & 1u) ? sc : -sc;
          const float ev = __fsub_rn(f4get(xv, c), so);
          acc = __fadd_rn(acc, __fmul_rn(ev, ev));
        }
      }
      acc = warp_butterfly_sum(acc);
      if (lane == 0) wsum[warp] = acc;
      __syncthreads();
      if (p == 0) {
        float* part = r < G.W ? ws.wpart + ((uint64_t)r * G.nc + tl.g) * G.tpc
                              : ws.spart + (uint64_t)tl.g * G.tpc;
        part[tl.t] = tree8(wsum);
      }
      __syncthreads();
    }
  }
}

}  // namespace

cudaError_t launch_error_norm(const MaterializeArgs& a, const Workspace& ws, int sms,
                              cudaStream_t s) {
  k_error_norm<<<grid_for(k_error_norm, sms, a.geo.n_tiles), kThreads, 0, s>>>(a, ws);
  return cudaGetLastError();
}

}  // namespace ob
