// Server side of the 1-bit compressed optimizer step: every server j
// averages the W workers' compressed chunks of its partition, adds its own
// error and compresses again (1-bit LAMB summary, paragraphs 3-4: the
// server error delta~ and the 3-phase Alltoall/AllGather exchange).
//
// Per element k of chunk g:
//   z    = (sum over w = 0..W-1, in order, from 0, of scale_w(g)*sign_w(k)) / W
//   e_s  = y_prev - sscale_prev*sign(y_prev)   (deferred server error)
//   y    = rho_l*e_s + z                        (1-bit Adam: e_s + z)
//   sbit = y >= 0; y is stored in place of e_s
//   sscale(g) = mean |y| over the chunk
//
// The workers' words are laid out worker-major ([W][n_pad/32]), so the
// W-way gather of one tile is W contiguous 512-byte runs; a CTA stages them
// in shared memory and every lane reads the four words it needs from there.
#include "ob_internal.cuh"

namespace ob {
namespace {

template <bool LAMB>
__global__ void __launch_bounds__(kThreads) k_server(const ServerArgs A) {
  __shared__ uint32_t sbw[OB_MAX_WORKERS * (kTile / 32)];
  __shared__ float sc[OB_MAX_WORKERS];
  __shared__ float ws[8];
  __shared__ int s_last;
  const Geo& G = A.geo;
  const int p = threadIdx.x, lane = p & 31, warp = p >> 5;
  const float fW = (float)G.W;

  for (uint32_t T = blockIdx.x; T < G.n_tiles; T += gridDim.x) {
    const Tile tl = decode_tile(G, T);
    const uint32_t nw = tl.len / 32;
    const uint64_t word0 = tl.start >> 5;
    if ((uint32_t)p < G.W) sc[p] = __ldcg(A.scales + (uint64_t)p * G.nc + tl.g);
    for (uint32_t idx = p; idx < G.W * nw; idx += kThreads) {
      uint32_t w = idx / nw, q = idx - w * nw;
      sbw[w * (kTile / 32) + q] = __ldcs(A.bits + (uint64_t)w * G.words + word0 + q);
    }
    const float osc = __ldcg(A.sscales + tl.g);
    __syncthreads();

    float acc = 0.0f;
    uint32_t l = 0;
    uint64_t lend = 0;
    float r_l = 1.0f;
    if constexpr (LAMB) {
      l = __ldg(A.ws.tile_layer + T);
      lend = __ldg(A.ws.layer_off + l + 1);
      r_l = A.ratio_ef ? __fdiv_rn(__ldg(A.c_prev2 + l), __ldg(A.c_prev + l)) : 1.0f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t off = 1024u * i + 4u * p;
      const bool valid = off < tl.len;
      const uint64_t k0 = tl.start + off;
      float4 ev = make_float4(0.f, 0.f, 0.f, 0.f);
      uint32_t owd = 0;
      float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (valid) {
        ev = __ldcs(reinterpret_cast<const float4*>(A.e_s + k0));
        owd = A.sbits[k0 >> 5];
        const uint32_t widx = off >> 5;
        const int sh = 4 * (p & 7);
        for (uint32_t w = 0; w < G.W; ++w) {
          const uint32_t wd = sbw[w * (kTile / 32) + widx] >> sh;
          const float s = sc[w];
#pragma unroll
          for (int c = 0; c < 4; ++c) z[c] = __fadd_rn(z[c], ((wd >> c) & 1u) ? s : -s);
        }
      }
      float4 yv;
      uint32_t nib = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint64_t k = k0 + c;
        float y = 0.0f;
        if (valid && k < G.n) {
          const float zc = __fdiv_rn(z[c], fW);
          const int sh = 4 * (p & 7) + c;
          const float so = ((owd >> sh) & 1u) ? osc : -osc;
          const float et = __fsub_rn(f4at(ev, c), so);
          if constexpr (LAMB) {
            if (advance_layer(A.ws.layer_off, G.L, k, l, lend))
              r_l = A.ratio_ef ? __fdiv_rn(__ldg(A.c_prev2 + l), __ldg(A.c_prev + l)) : 1.0f;
            y = __fadd_rn(__fmul_rn(r_l, et), zc);
          } else {
            y = __fadd_rn(et, zc);
          }
          acc = __fadd_rn(acc, fabsf(y));
          if (y >= 0.0f) nib |= 1u << c;
        }
        f4at(yv, c) = y;
      }
      const uint32_t word = pack_word(nib, lane);
      if (valid) {
        __stcs(reinterpret_cast<float4*>(A.e_s + k0), yv);
        if ((p & 7) == 0) A.sbits[k0 >> 5] = word;
      }
    }
    acc = warp_butterfly_sum(acc);
    if (lane == 0) ws[warp] = acc;
    __syncthreads();
    if (p == 0) A.ws.spart[(uint64_t)tl.g * G.tpc + tl.t] = tree8(ws);
    __threadfence();
    __syncthreads();
    if (p == 0) {
      unsigned prev = atomicAdd(A.ws.scnt + tl.g, 1u);
      s_last = (prev == tl.ntc - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      if (warp == 0) {
        float sum = ordered_sum(A.ws.spart + (uint64_t)tl.g * G.tpc, tl.ntc, lane);
        if (lane == 0) {
          A.sscales[tl.g] = mean_of(sum, tl.real);
          A.ws.scnt[tl.g] = 0u;
        }
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_server(const ServerArgs& a, bool lamb, int sms, cudaStream_t s) {
  if (lamb) {
    k_server<true><<<grid_for(k_server<true>, sms, a.geo.n_tiles), kThreads, 0, s>>>(a);
  } else {
    k_server<false><<<grid_for(k_server<false>, sms, a.geo.n_tiles), kThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace ob
