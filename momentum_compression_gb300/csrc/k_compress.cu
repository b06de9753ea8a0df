// Worker compression of the 1-bit compressed optimizer step, all W workers
// in one pass over the fused buffer.
//
// Per element k of worker w ("1bit Adam" write-up, 2.1; gradient
// quantization tutorial, "1-bit 梯度量化"; 1-bit LAMB summary, paragraphs
// 2-3):
//   e_w   = x_prev - scale_prev*sign(x_prev)   (the deferred error of the
//           previous step, rebuilt from the stored x, bits and scale)
//   m_w   = b1*m + (1-b1)*g_w
//   x     = sigma_l*m_w + rho_l*e_w            (1-bit Adam: m_w + e_w)
//   bit   = x >= 0; x is stored in place of e_w
//   scale(chunk) = mean |x| over the chunk (finalised by the last CTA of
//   the chunk to arrive)
//
// One CTA of 256 threads owns one tile of 4096 elements and all W workers
// of it, so the momentum m is read once per element.  Lane p handles
// elements 1024*i + 4*p + c (i, c = 0..3) with 128-bit loads; that is also
// the fixed summation order of the tile total.  Signs are packed with
// three xor-shuffles per 32-bit word.  No device-side wait: the chunk scale
// is finalised by whichever CTA brings the chunk's arrival count to its
// tile count.
#include "ob_internal.cuh"

namespace ob {
namespace {

template <bool BF16, bool LAMB>
__global__ void __launch_bounds__(kThreads)
    k_compress(const CompressArgs A) {
  __shared__ float ws[OB_MAX_WORKERS][8];
  __shared__ int s_last;
  const Geo& G = A.geo;
  const int p = threadIdx.x, lane = p & 31, warp = p >> 5;
  const float b1 = A.b1, ob1 = A.ob1;

  for (uint32_t T = blockIdx.x; T < G.n_tiles; T += gridDim.x) {
    const Tile tl = decode_tile(G, T);

    float4 mv[4];
    bool valid[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t off = 1024u * i + 4u * p;
      valid[i] = off < tl.len;
      if (valid[i]) mv[i] = __ldcs(reinterpret_cast<const float4*>(A.m + tl.start + off));
      else mv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // Per-element layer factors (1-bit LAMB only).
    float sig[4][4], rho[4][4];
    if constexpr (LAMB) {
      uint32_t l = __ldg(A.ws.tile_layer + T);
      uint64_t lend = __ldg(A.ws.layer_off + l + 1);
      float s_l = __ldg(A.s + l);
      float r_l = A.ratio_ef ? __fdiv_rn(__ldg(A.c_prev2 + l), __ldg(A.c_prev + l)) : 1.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint64_t k = tl.start + 1024u * i + 4u * p + c;
          if (valid[i] && k < G.n &&
              advance_layer(A.ws.layer_off, G.L, k, l, lend)) {
            s_l = __ldg(A.s + l);
            r_l = A.ratio_ef ? __fdiv_rn(__ldg(A.c_prev2 + l), __ldg(A.c_prev + l)) : 1.0f;
          }
          sig[i][c] = s_l;
          rho[i][c] = r_l;
        }
    }

    for (uint32_t w = 0; w < G.W; ++w) {
      const float osc = __ldcg(A.scales + (uint64_t)w * G.nc + tl.g);
      float* __restrict__ e = A.e[w];
      uint32_t* __restrict__ bw = A.bits + (uint64_t)w * G.words;
      float acc = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint64_t k0 = tl.start + 1024u * i + 4u * p;
        float4 gv = make_float4(0.f, 0.f, 0.f, 0.f), ev = gv;
        uint32_t owd = 0;
        if (valid[i]) {
          gv = load_grad4<BF16>(A.g[w], k0);
          ev = __ldcs(reinterpret_cast<const float4*>(e + k0));
          owd = bw[k0 >> 5];
        }
        float4 xv;
        uint32_t nib = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint64_t k = k0 + c;
          float x = 0.0f;
          if (valid[i] && k < G.n) {
            const int sh = 4 * (p & 7) + c;
            const float so = ((owd >> sh) & 1u) ? osc : -osc;  // scale*sign
            const float et = __fsub_rn(f4at(ev, c), so);
            const float mw = __fadd_rn(__fmul_rn(b1, f4at(mv[i], c)),
                                       __fmul_rn(ob1, f4at(gv, c)));
            if constexpr (LAMB) {
              x = __fadd_rn(__fmul_rn(sig[i][c], mw), __fmul_rn(rho[i][c], et));
            } else {
              x = __fadd_rn(mw, et);
            }
            acc = __fadd_rn(acc, fabsf(x));
            if (x >= 0.0f) nib |= 1u << c;
          }
          f4at(xv, c) = x;
        }
        const uint32_t word = pack_word(nib, lane);
        if (valid[i]) {
          __stcs(reinterpret_cast<float4*>(e + k0), xv);
          if ((p & 7) == 0) bw[k0 >> 5] = word;
        }
      }
      acc = warp_butterfly_sum(acc);
      if (lane == 0) ws[w][warp] = acc;
    }
    __syncthreads();
    if ((uint32_t)p < G.W) {
      A.ws.wpart[((uint64_t)p * G.nc + tl.g) * G.tpc + tl.t] = tree8(ws[p]);
    }
    __threadfence();
    __syncthreads();
    if (p == 0) {
      unsigned prev = atomicAdd(A.ws.wcnt + tl.g, 1u);
      s_last = (prev == tl.ntc - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      for (uint32_t w = warp; w < G.W; w += kThreads / 32) {
        float sum = ordered_sum(A.ws.wpart + ((uint64_t)w * G.nc + tl.g) * G.tpc,
                                tl.ntc, lane);
        if (lane == 0) A.scales[(uint64_t)w * G.nc + tl.g] = mean_of(sum, tl.real);
      }
      if (p == 0) A.ws.wcnt[tl.g] = 0u;
    }
    __syncthreads();
  }
}

}  // namespace

template <bool BF16, bool LAMB>
static cudaError_t run_compress(const CompressArgs& a, int sms, cudaStream_t s) {
  const int grid = grid_for(k_compress<BF16, LAMB>, sms, a.geo.n_tiles);
  k_compress<BF16, LAMB><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_compress(const CompressArgs& a, bool bf16, bool lamb, int sms,
                            cudaStream_t s) {
  if (bf16) return lamb ? run_compress<true, true>(a, sms, s) : run_compress<true, false>(a, sms, s);
  return lamb ? run_compress<false, true>(a, sms, s) : run_compress<false, false>(a, sms, s);
}

}  // namespace ob
