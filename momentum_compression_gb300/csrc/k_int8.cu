// Block-wise INT8 stochastic-rounding quantizer (gradient quantization
// tutorial, "FP32 → INT8 量化": scale = max|g|/127 per block, stochastic
// rounding; and its GradientQuantizeINT8 example: floor plus a Bernoulli
// draw on the fractional part, clamp to ±127).
//
// Each group of four elements draws one Philox4x32-10 output (four 32-bit
// words) from counter (k>>2, step), whichever lane quantises it.  Without
// error feedback half a warp takes a block of 256 elements (16 per lane);
// with it a warp does (8 per lane, in the order of the per-block error
// monitor's sums).  The block max is a (half-)warp max.
//
// Philox4x32-10 is in philox.cuh.
#include "ob_internal.cuh"
#include "philox.cuh"
#include "sround.cuh"

namespace ob {
namespace {

// Quantizes two groups of 4 values, xv[h] (h = 0, 1; elements 4*grp[h] ..
// 4*grp[h]+3), one Philox output per group, both drawn side by side; dq[h]
// receives q*scale and packed[h] the four codes.  rcp: code_rcp(scale)
// (sround.cuh): the codes come from code_fast where certain, else from
// code_exact (for all 8 values of a lane that has an uncertain one; the
// two agree wherever code_fast is certain).  Every lane of the warp calls
// it (the fallback is taken by vote); values beyond the tensor are 0 and
// code as 0.
__device__ __forceinline__ void quant8(const float4 (&xv)[2], float scale, float rcp,
                                       const uint64_t (&grp)[2], uint64_t step,
                                       const PhiloxKeys& K, float4 (&dq)[2],
                                       uint32_t (&packed)[2]) {
  uint4 rnd[2];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    rnd[h] = make_uint4((uint32_t)grp[h], (uint32_t)(grp[h] >> 32), (uint32_t)step,
                        (uint32_t)(step >> 32));
  philox4x32_10_x2(rnd[0], rnd[1], K);
  float qf[2][4], u[2][4];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int c = 0; c < 4; ++c) u[h][c] = uniform_of(word_of(rnd[h], c));
  if (rcp != 0.0f) {
    bool unsure = false;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        bool certain;
        qf[h][c] = code_fast<127>(f4get(xv[h], c), rcp, u[h][c], &certain);
        unsure |= !certain;
      }
    // the definition where code_fast is not certain
    if (__any_sync(kFull, unsure) && unsure) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 4; ++c) qf[h][c] = code_exact<127>(f4get(xv[h], c), scale, u[h][c]);
    }
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        qf[h][c] = scale != 0.0f ? code_exact<127>(f4get(xv[h], c), scale, u[h][c]) : 0.0f;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    packed[h] = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      f4at(dq[h], c) = __fmul_rn(qf[h][c], scale);
      packed[h] |= ((uint32_t)(int32_t)qf[h][c] & 0xffu) << (8 * c);
    }
  }
}

// Quantizes the 4 values x of group `grp` (elements 4*grp .. 4*grp+3);
// dq receives q*scale.  rcp: code_rcp(scale) (sround.cuh): the codes come
// from code_fast where certain, else from code_exact.  Every lane
// of the warp calls it (the fallback is taken by vote); values beyond the
// tensor are 0 and code as 0.
__device__ __forceinline__ uint32_t quant4(const float4& xv, float scale, float rcp,
                                           uint64_t grp, uint64_t step, const PhiloxKeys& K,
                                           float4& dq) {
  const uint4 ctr = make_uint4((uint32_t)grp, (uint32_t)(grp >> 32), (uint32_t)step,
                               (uint32_t)(step >> 32));
  const uint4 rnd = philox4x32_10(ctr, K);
  float qf[4], u[4];
  bool unsure = false;
  if (rcp != 0.0f) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      u[c] = uniform_of(word_of(rnd, c));
      bool certain;
      qf[c] = code_fast<127>(f4get(xv, c), rcp, u[c], &certain);
      unsure |= !certain;
    }
    // the definition where code_fast is not certain
    if (__any_sync(kFull, unsure) && unsure) {
#pragma unroll
      for (int c = 0; c < 4; ++c) qf[c] = code_exact<127>(f4get(xv, c), scale, u[c]);
    }
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      qf[c] = scale != 0.0f ? code_exact<127>(f4get(xv, c), scale, uniform_of(word_of(rnd, c)))
                            : 0.0f;
  }
  uint32_t packed = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    f4at(dq, c) = __fmul_rn(qf[c], scale);
    packed |= ((uint32_t)(int32_t)qf[c] & 0xffu) << (8 * c);
  }
  return packed;
}

// Loads the two 4-element groups lane `lane` owns in block b (zeros and a
// valid count of 0..4 per group beyond n).
__device__ __forceinline__ void load_block(const float* __restrict__ g, uint64_t n, uint64_t b,
                                           int lane, float4 (&gv)[2], int (&nv)[2]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint64_t k = b * 256 + 128 * h + 4 * lane;
    nv[h] = k >= n ? 0 : (n - k >= 4 ? 4 : (int)(n - k));
    if (nv[h] == 4) {
      gv[h] = *reinterpret_cast<const float4*>(g + k);
    } else {
      gv[h] = make_float4(nv[h] > 0 ? g[k] : 0.f, nv[h] > 1 ? g[k + 1] : 0.f,
                          nv[h] > 2 ? g[k + 2] : 0.f, 0.f);
    }
  }
}

__device__ __forceinline__ void store4(float* __restrict__ dst, uint64_t k, int nv,
                                       const float4& v) {
  if (nv == 4) {
    *reinterpret_cast<float4*>(dst + k) = v;
  } else {
#pragma unroll
    for (int c = 0; c < 3; ++c)
      if (c < nv) dst[k + c] = f4get(v, c);
  }
}

// DEQ: write q*scale.  EF: error feedback -- x = g + e is quantised and
// e := x - q*scale.  ERR2: per-block sum of the squared residual (lane j
// adds its 8 squares in element order, then a warp butterfly).
// With error feedback: one warp per block, lane j holding elements 4j ..
// 4j+3 and 128+4j .. 128+4j+3 (the next block's loads in flight while this
// one is quantised); x = g + e is quantised and e := x - q*scale.  The two
// halves' Philox outputs are drawn one at a time (quant4): side by side
// (quant8) their registers cost a CTA per SM and measured 6.4% slower.
template <bool DEQ, bool ERR2>
__device__ __forceinline__ void quant_int8_ef_body(const float* __restrict__ g,
                                                   float* __restrict__ e, uint64_t n,
                                                   int8_t* __restrict__ q,
                                                   float* __restrict__ scales,
                                                   const PhiloxKeys& K, uint64_t step,
                                                   float* __restrict__ deq,
                                                   float* __restrict__ err2) {
  const int lane = threadIdx.x & 31;
  const uint64_t nblk = (n + 255) / 256;
  const uint64_t warps = (uint64_t)gridDim.x * (kThreads / 32);
  uint64_t b = (uint64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  float4 gv[2], ev[2];
  int nv[2];
  if (b < nblk) {
    load_block(g, n, b, lane, gv, nv);
    load_block(e, n, b, lane, ev, nv);
  }
  for (; b < nblk; b += warps) {
    float4 gn[2], en[2];
    int nn[2] = {0, 0};
    if (b + warps < nblk) {
      load_block(g, n, b + warps, lane, gn, nn);
      load_block(e, n, b + warps, lane, en, nn);
    }
    float4 xv[2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
      xv[h] = make_float4(__fadd_rn(gv[h].x, ev[h].x), __fadd_rn(gv[h].y, ev[h].y),
                          __fadd_rn(gv[h].z, ev[h].z), __fadd_rn(gv[h].w, ev[h].w));
    // fmaxf returns the other operand when one is NaN: a NaN never wins
    float mx = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (c < nv[h]) mx = fmaxf(mx, fabsf(f4get(xv[h], c)));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    const float scale = mx == 0.0f ? 0.0f : __fdiv_rn(mx, 127.0f);
    // 1/scale for the division-free codes (quant4); a scale below the
    // normal range takes the definition for every value
    const float rcp = code_rcp(scale);
    if (lane == 0) scales[b] = scale;
    float acc2 = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint64_t k = b * 256 + 128 * h + 4 * lane;
      // every lane quantises (values beyond the tensor are 0 and code as 0)
      float4 dq = make_float4(0.f, 0.f, 0.f, 0.f);
      const uint32_t packed = quant4(xv[h], scale, rcp, k >> 2, step, K, dq);
      if (nv[h] > 0) {
        if (nv[h] == 4) {
          *reinterpret_cast<uint32_t*>(q + k) = packed;
        } else {
#pragma unroll
          for (int c = 0; c < 3; ++c)
            if (c < nv[h]) q[k + c] = (int8_t)((packed >> (8 * c)) & 0xffu);
        }
        if constexpr (DEQ) store4(deq, k, nv[h], dq);
      }
      float4 r;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        f4at(r, c) = __fsub_rn(f4get(xv[h], c), f4get(dq, c));
        if (ERR2 && c < nv[h]) acc2 = __fadd_rn(acc2, __fmul_rn(f4get(r, c), f4get(r, c)));
      }
      if (nv[h] > 0) store4(e, k, nv[h], r);
    }
    if constexpr (ERR2) {
      acc2 = warp_butterfly_sum(acc2);
      if (lane == 0) err2[b] = acc2;
    }
    gv[0] = gn[0];
    gv[1] = gn[1];
    ev[0] = en[0];
    ev[1] = en[1];
    nv[0] = nn[0];
    nv[1] = nn[1];
  }
}

// Without error feedback: half a warp per block.  Lanes 16h .. 16h+15 take
// block 2*pair + h, and lane j = lane % 16 holds elements 64r + 4j ..
// 64r + 4j + 3 (r = 0..3) of it -- four 128-bit loads, 256 contiguous bytes
// per half-warp and row -- so the block max, the scale and its reciprocal
// are paid once per 16 values, and the four Philox outputs are drawn in two
// side-by-side pairs.  The next pair's loads are in flight while this one is
// quantised (3 CTAs per SM, 79 registers: 2.3% faster than without them at
// 4).  (The error-feedback forms keep a warp per block: the per-block error
// monitor's order is lane j's 8 values, then the warp.)
template <bool DEQ>
__global__ void __launch_bounds__(kThreads, 3)
    k_quant_int8(const float* __restrict__ g, uint64_t n, int8_t* __restrict__ q,
                 float* __restrict__ scales, const PhiloxKeys K, uint64_t step,
                 float* __restrict__ deq) {
  const int lane = threadIdx.x & 31, j = lane & 15, half = lane >> 4;
  const uint64_t nblk = (n + 255) / 256;
  const uint64_t npair = (nblk + 1) / 2;
  const uint64_t warps = (uint64_t)gridDim.x * (kThreads / 32);
  // lane j's 16 values of block b (b == nblk for the missing second block
  // of an odd count: every value lies beyond n there, codes as 0 and is not
  // stored)
  auto load_block16 = [&](uint64_t b, float4 (&xv)[4], int (&nv)[4]) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint64_t k = b * 256 + 64 * r + 4 * j;
      nv[r] = k >= n ? 0 : (n - k >= 4 ? 4 : (int)(n - k));
      if (nv[r] == 4) {
        xv[r] = *reinterpret_cast<const float4*>(g + k);
      } else {
        xv[r] = make_float4(nv[r] > 0 ? g[k] : 0.f, nv[r] > 1 ? g[k + 1] : 0.f,
                            nv[r] > 2 ? g[k + 2] : 0.f, 0.f);
      }
    }
  };
  uint64_t pr = (uint64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  float4 xn[4];
  int nn[4] = {0, 0, 0, 0};
  if (pr < npair) load_block16(2 * pr + half, xn, nn);
  for (; pr < npair; pr += warps) {
    const uint64_t b = 2 * pr + half;
    float4 xv[4];
    int nv[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      xv[r] = xn[r];
      nv[r] = nn[r];
    }
    if (pr + warps < npair) load_block16(2 * (pr + warps) + half, xn, nn);
    // fmaxf returns the other operand when one is NaN: a NaN never wins
    float mx = 0.0f;
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (c < nv[r]) mx = fmaxf(mx, fabsf(f4get(xv[r], c)));
    // the half-warp's max (xor offsets below 16 stay inside the half)
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    const float scale = mx == 0.0f ? 0.0f : __fdiv_rn(mx, 127.0f);
    const float rcp = code_rcp(scale);
    if (j == 0 && b < nblk) scales[b] = scale;
#pragma unroll
    for (int rp = 0; rp < 2; ++rp) {
      const float4 xp[2] = {xv[2 * rp], xv[2 * rp + 1]};
      const uint64_t k0 = b * 256 + 128 * rp + 4 * j;
      const uint64_t grp[2] = {k0 >> 2, (k0 + 64) >> 2};
      float4 dqv[2];
      uint32_t pk[2];
      quant8(xp, scale, rcp, grp, step, K, dqv, pk);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = 2 * rp + h;
        const uint64_t k = k0 + 64 * h;
        if (nv[r] > 0) {
          if (nv[r] == 4) {
            *reinterpret_cast<uint32_t*>(q + k) = pk[h];
          } else {
#pragma unroll
            for (int c = 0; c < 3; ++c)
              if (c < nv[r]) q[k + c] = (int8_t)((pk[h] >> (8 * c)) & 0xffu);
          }
          if constexpr (DEQ) store4(deq, k, nv[r], dqv[h]);
        }
      }
    }
  }
}

template <bool DEQ, bool ERR2>
__global__ void __launch_bounds__(kThreads)
    k_quant_int8_ef(const float* __restrict__ g, float* __restrict__ e, uint64_t n,
                    int8_t* __restrict__ q, float* __restrict__ scales, const PhiloxKeys K,
                    uint64_t step, float* __restrict__ deq, float* __restrict__ err2) {
  quant_int8_ef_body<DEQ, ERR2>(g, e, n, q, scales, K, step, deq, err2);
}

template <bool DEQ, bool EF, bool ERR2>
cudaError_t run_int8(const float* g, float* e, uint64_t n, int8_t* q, float* scales,
                     uint64_t seed, uint64_t step, float* deq, float* err2, int sms,
                     cudaStream_t s) {
  const uint64_t nblk = (n + 255) / 256;
  const uint64_t ctas = (nblk + kThreads / 32 - 1) / (kThreads / 32);
  // the round keys go in as a kernel parameter (see philox.cuh)
  const PhiloxKeys K = philox_keys((uint32_t)seed, (uint32_t)(seed >> 32));
  if constexpr (EF) {
    k_quant_int8_ef<DEQ, ERR2><<<grid_for(k_quant_int8_ef<DEQ, ERR2>, sms, ctas), kThreads, 0,
                                 s>>>(g, e, n, q, scales, K, step, deq, err2);
  } else {
    const uint64_t pctas = ((nblk + 1) / 2 + kThreads / 32 - 1) / (kThreads / 32);
    k_quant_int8<DEQ><<<grid_for(k_quant_int8<DEQ>, sms, pctas), kThreads, 0, s>>>(
        g, n, q, scales, K, step, deq);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_int8(const float* g, uint64_t n, int8_t* q, float* scales,
                              uint64_t seed, uint64_t step, float* deq, int sms,
                              cudaStream_t s) {
  if (deq) return run_int8<true, false, false>(g, nullptr, n, q, scales, seed, step, deq,
                                               nullptr, sms, s);
  return run_int8<false, false, false>(g, nullptr, n, q, scales, seed, step, nullptr, nullptr,
                                       sms, s);
}

cudaError_t launch_quant_int8_ef(const float* g, float* e, uint64_t n, int8_t* q, float* scales,
                                 uint64_t seed, uint64_t step, float* deq, float* err2, int sms,
                                 cudaStream_t s) {
  if (deq) {
    return err2 ? run_int8<true, true, true>(g, e, n, q, scales, seed, step, deq, err2, sms, s)
                : run_int8<true, true, false>(g, e, n, q, scales, seed, step, deq, err2, sms, s);
  }
  return err2 ? run_int8<false, true, true>(g, e, n, q, scales, seed, step, deq, err2, sms, s)
              : run_int8<false, true, false>(g, e, n, q, scales, seed, step, deq, err2, sms, s);
}

}  // namespace ob
