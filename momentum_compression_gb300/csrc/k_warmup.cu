// Uncompressed warmup steps and the switch to compression.
//
// The "1bit Adam" write-up (6, tuning) and the gradient quantization
// tutorial ("预热训练") run the first steps at full precision; the 1-bit
// LAMB summary (paragraph 1) freezes v at the end of warmup and keeps the
// warmup average c_avg of LAMB's coefficient, and (paragraph 2) fixes a
// per-layer momentum scale from the momentum norms at that point.
//
//   g_bar = (sum over w, in order, from 0, of g_w) / W
//   m = b1*m + (1-b1)*g_bar;  v = b2*v + (1-b2)*g_bar^2
//   Adam:  p = p - lr*(m/(sqrt(v)+eps))
//   LAMB:  u = m/(sqrt(v)+eps); c_l = clip(||p_l||/||u_l||, c_min, c_max)
//          (1 if a norm is 0); p = p - (lr*c_l)*u
//   begin: rms_l = ||m_l||/sqrt(n_l); s_l = mean(rms)/rms_l;
//          c_avg = c_sum/T_w; r_prev = 1; c_prev = c_prev2 = c_avg
//
// Layer norms use the fixed tile order counted from each layer's own
// start, so those kernels walk "layer tiles" with scalar loads (a layer may
// start at any element).
#include "ob_internal.cuh"

namespace ob {
namespace {

template <bool BF16>
__device__ __forceinline__ float load_grad1(const void* g, uint64_t k) {
  if constexpr (BF16) return bf16_to_f32(__ldcs(static_cast<const unsigned short*>(g) + k));
  else return __ldcs(static_cast<const float*>(g) + k);
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads) k_warmup_adam(const WarmupArgs A) {
  const Geo& G = A.geo;
  const int p = threadIdx.x;
  for (uint32_t T = blockIdx.x; T < G.n_tiles; T += gridDim.x) {
    const Tile tl = decode_tile(G, T);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t off = 1024u * i + 4u * p;
      if (off >= tl.len) continue;
      const uint64_t k0 = tl.start + off;
      if (k0 >= G.n) {
        __stcs(reinterpret_cast<float4*>(A.m + k0), make_float4(0.f, 0.f, 0.f, 0.f));
        continue;
      }
      float4 gb = make_float4(0.f, 0.f, 0.f, 0.f);
      for (uint32_t w = 0; w < G.W; ++w) {
        const float4 gv = load_grad4<BF16>(A.g[w], k0);
        gb.x = __fadd_rn(gb.x, gv.x);
        gb.y = __fadd_rn(gb.y, gv.y);
        gb.z = __fadd_rn(gb.z, gv.z);
        gb.w = __fadd_rn(gb.w, gv.w);
      }
      float4 mv = __ldcs(reinterpret_cast<const float4*>(A.m + k0));
      float4 vv = __ldcs(reinterpret_cast<const float4*>(A.v + k0));
      float4 pv = __ldcs(reinterpret_cast<const float4*>(A.p + k0));
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (k0 + c >= G.n) {
          f4at(mv, c) = 0.0f;
          continue;
        }
        const float g = div_by_workers(f4at(gb, c), A.fW, A.inv_w);
        const float m = __fadd_rn(__fmul_rn(A.b1, f4at(mv, c)), __fmul_rn(A.ob1, g));
        const float v = __fadd_rn(__fmul_rn(A.b2, f4at(vv, c)),
                                  __fmul_rn(A.ob2, __fmul_rn(g, g)));
        const float d = __fadd_rn(__fsqrt_rn(v), A.eps);
        const float u = __fdiv_rn(m, d);
        f4at(mv, c) = m;
        f4at(vv, c) = v;
        f4at(pv, c) = __fsub_rn(f4at(pv, c), __fmul_rn(A.lr, u));
      }
      __stcs(reinterpret_cast<float4*>(A.m + k0), mv);
      __stcs(reinterpret_cast<float4*>(A.v + k0), vv);
      __stcs(reinterpret_cast<float4*>(A.p + k0), pv);
    }
  }
}

// Layer tile LT -> (layer, tile inside the layer, first element, length).
struct LTile {
  uint32_t l, t, len;
  uint64_t start;
};

__device__ __forceinline__ LTile decode_ltile(const Workspace& ws, uint32_t L, uint32_t LT) {
  uint32_t lo = 0, hi = L;  // pref[lo] <= LT < pref[hi]
  while (hi - lo > 1) {
    uint32_t mid = (lo + hi) >> 1;
    if (__ldg(ws.ltile_pref + mid) <= LT) lo = mid; else hi = mid;
  }
  LTile r;
  r.l = lo;
  r.t = LT - __ldg(ws.ltile_pref + lo);
  const uint64_t a = __ldg(ws.layer_off + lo), b = __ldg(ws.layer_off + lo + 1);
  r.start = a + (uint64_t)r.t * kTile;
  const uint64_t left = b - r.start;
  r.len = (uint32_t)(left < kTile ? left : kTile);
  return r;
}

// Block total of two lane sums in the fixed order; valid in thread 0.
__device__ __forceinline__ void block_sum2(float a, float b, float (*ws)[8], float& ta,
                                           float& tb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_butterfly_sum(a);
  b = warp_butterfly_sum(b);
  if (lane == 0) {
    ws[0][warp] = a;
    ws[1][warp] = b;
  }
  __syncthreads();
  ta = tree8(ws[0]);
  tb = tree8(ws[1]);
}

// Sums of the squares staged in shared memory in the fixed lane order:
// lane p adds elements 1024*i + 4*p + c (i, c = 0..3) from 0.  Entries past
// the tile's end hold +0, which leaves a non-negative sum unchanged.
__device__ __forceinline__ float lane_sum_sq(const float* sq, int p) {
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 v = *reinterpret_cast<const float4*>(sq + 1024 * i + 4 * p);
    acc = __fadd_rn(acc, v.x);
    acc = __fadd_rn(acc, v.y);
    acc = __fadd_rn(acc, v.z);
    acc = __fadd_rn(acc, v.w);
  }
  return acc;
}

// LAMB warmup, pass A: per layer tile (counted from the layer's start) the
// elementwise update of m and v, and the tile totals of p^2 and u^2 for the
// layer norms.  Threads read and write element t + 256*j (coalesced), stage
// the squares in shared memory and sum them there in the fixed lane order.
template <bool BF16>
__global__ void __launch_bounds__(kThreads) k_warmup_lamb_a(const WarmupArgs A) {
  __shared__ __align__(16) float sp[kTile];
  __shared__ __align__(16) float su[kTile];
  __shared__ float ws[2][8];
  const Geo& G = A.geo;
  const int p = threadIdx.x;
  for (uint32_t LT = blockIdx.x; LT < G.n_ltiles; LT += gridDim.x) {
    const LTile lt = decode_ltile(A.ws, G.L, LT);
    float lp, lu;  // this lane's sums of p^2 and u^2 in the fixed order
    if ((lt.start & 3) == 0) {
      // the layer tile starts on a 16-byte boundary: lane p loads elements
      // 1024*i + 4*p .. +3 with 128-bit loads -- exactly the elements it
      // adds, in the order it adds them, so no staging is needed.  A last
      // group that runs past the layer's end is stored element by element
      // (the rest belongs to the next layer).
      lp = 0.0f;
      lu = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t off = 1024u * i + 4u * p;
        if (off >= lt.len) continue;
        const uint64_t k0 = lt.start + off;
        const uint32_t nv = lt.len - off < 4u ? lt.len - off : 4u;
        float4 gb = make_float4(0.f, 0.f, 0.f, 0.f);
        for (uint32_t w = 0; w < G.W; ++w) {
          const float4 gv = load_grad4<BF16>(A.g[w], k0);
          gb.x = __fadd_rn(gb.x, gv.x);
          gb.y = __fadd_rn(gb.y, gv.y);
          gb.z = __fadd_rn(gb.z, gv.z);
          gb.w = __fadd_rn(gb.w, gv.w);
        }
        float4 mv = __ldcs(reinterpret_cast<const float4*>(A.m + k0));
        float4 vv = __ldcs(reinterpret_cast<const float4*>(A.v + k0));
        const float4 pv = __ldcs(reinterpret_cast<const float4*>(A.p + k0));
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if ((uint32_t)c >= nv) continue;
          const float g = div_by_workers(f4at(gb, c), A.fW, A.inv_w);
          const float m = __fadd_rn(__fmul_rn(A.b1, f4at(mv, c)), __fmul_rn(A.ob1, g));
          const float v = __fadd_rn(__fmul_rn(A.b2, f4at(vv, c)),
                                    __fmul_rn(A.ob2, __fmul_rn(g, g)));
          const float u = __fdiv_rn(m, __fadd_rn(__fsqrt_rn(v), A.eps));
          f4at(mv, c) = m;
          f4at(vv, c) = v;
          lp = __fadd_rn(lp, __fmul_rn(f4get(pv, c), f4get(pv, c)));
          lu = __fadd_rn(lu, __fmul_rn(u, u));
        }
        if (nv == 4) {
          __stcs(reinterpret_cast<float4*>(A.m + k0), mv);
          __stcs(reinterpret_cast<float4*>(A.v + k0), vv);
        } else {
          for (uint32_t c = 0; c < nv; ++c) {
            A.m[k0 + c] = f4at(mv, c);
            A.v[k0 + c] = f4at(vv, c);
          }
        }
      }
    } else {
      // any other start: coalesced scalar accesses (thread t takes elements
      // t + 256*j), the squares staged in shared memory at their tile
      // positions and summed there in the fixed lane order
#pragma unroll 4
      for (int j = 0; j < 16; ++j) {
        const uint32_t idx = p + kThreads * j;
        float pq = 0.0f, uq = 0.0f;
        if (idx < lt.len) {
          const uint64_t k = lt.start + idx;
          float gb = 0.0f;
          for (uint32_t w = 0; w < G.W; ++w) gb = __fadd_rn(gb, load_grad1<BF16>(A.g[w], k));
          gb = div_by_workers(gb, A.fW, A.inv_w);
          const float m = __fadd_rn(__fmul_rn(A.b1, A.m[k]), __fmul_rn(A.ob1, gb));
          const float v =
              __fadd_rn(__fmul_rn(A.b2, A.v[k]), __fmul_rn(A.ob2, __fmul_rn(gb, gb)));
          const float u = __fdiv_rn(m, __fadd_rn(__fsqrt_rn(v), A.eps));
          A.m[k] = m;
          A.v[k] = v;
          const float pk = __ldcs(A.p + k);
          pq = __fmul_rn(pk, pk);
          uq = __fmul_rn(u, u);
        }
        sp[idx] = pq;
        su[idx] = uq;
      }
      __syncthreads();
      lp = lane_sum_sq(sp, p);
      lu = lane_sum_sq(su, p);
    }
    float tp, tu;
    block_sum2(lp, lu, ws, tp, tu);
    if (p == 0) {
      A.ws.lpart[LT] = tp;
      A.ws.lpart[G.n_ltiles + LT] = tu;
    }
    __syncthreads();
  }
}

// LAMB warmup: per layer (one warp each) the norms ||p_l||, ||u_l|| from
// the tile totals in order, c = clip(||p||/||u||, c_min, c_max) (1 if a norm
// is 0); c_t = c, c_sum += c.
__global__ void __launch_bounds__(kThreads) k_warmup_lamb_c(const WarmupArgs A) {
  const Geo& G = A.geo;
  const int lane = threadIdx.x & 31;
  for (uint32_t l = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); l < G.L;
       l += gridDim.x * (kThreads / 32)) {
    const uint32_t b = __ldg(A.ws.ltile_pref + l);
    const uint32_t ntl = __ldg(A.ws.ltile_pref + l + 1) - b;
    const float np = __fsqrt_rn(ordered_sum(A.ws.lpart + b, ntl, lane));
    const float nu = __fsqrt_rn(ordered_sum(A.ws.lpart + G.n_ltiles + b, ntl, lane));
    if (lane == 0) {
      float c;
      if (np == 0.0f || nu == 0.0f) {
        c = 1.0f;
      } else {
        c = __fdiv_rn(np, nu);
        c = fmin_plain(fmax_plain(c, A.c_min), A.c_max);
      }
      A.ls.c_t[l] = c;
      A.ls.c_sum[l] = __fadd_rn(A.ls.c_sum[l], c);
    }
  }
}

__global__ void __launch_bounds__(kThreads) k_warmup_lamb_b(const WarmupArgs A) {
  const Geo& G = A.geo;
  const int p = threadIdx.x;
  for (uint32_t T = blockIdx.x; T < G.n_tiles; T += gridDim.x) {
    const Tile tl = decode_tile(G, T);
    uint32_t l = __ldg(A.ws.tile_layer + T);
    uint64_t lend = __ldg(A.ws.layer_off + l + 1);
    float t1 = __fmul_rn(A.lr, __ldcg(A.ls.c_t + l));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t off = 1024u * i + 4u * p;
      if (off >= tl.len) continue;
      const uint64_t k0 = tl.start + off;
      if (k0 >= G.n) {
        __stcs(reinterpret_cast<float4*>(A.m + k0), make_float4(0.f, 0.f, 0.f, 0.f));
        continue;
      }
      float4 mv = __ldcs(reinterpret_cast<const float4*>(A.m + k0));
      const float4 vv = __ldcs(reinterpret_cast<const float4*>(A.v + k0));
      float4 pv = __ldcs(reinterpret_cast<const float4*>(A.p + k0));
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint64_t k = k0 + c;
        if (k >= G.n) {
          f4at(mv, c) = 0.0f;
          continue;
        }
        if (advance_layer(A.ws.layer_off, G.L, k, l, lend))
          t1 = __fmul_rn(A.lr, __ldcg(A.ls.c_t + l));
        const float u = __fdiv_rn(f4at(mv, c), __fadd_rn(__fsqrt_rn(f4get(vv, c)), A.eps));
        f4at(pv, c) = __fsub_rn(f4at(pv, c), __fmul_rn(t1, u));
      }
      if (k0 + 3 >= G.n) __stcs(reinterpret_cast<float4*>(A.m + k0), mv);
      __stcs(reinterpret_cast<float4*>(A.p + k0), pv);
    }
  }
}

// End of warmup, pass 1: per layer tile the total of m^2 (coalesced loads,
// fixed lane order from shared memory, as in k_warmup_lamb_a).
__global__ void __launch_bounds__(kThreads) k_lamb_begin_tiles(const WarmupArgs A) {
  __shared__ __align__(16) float sq[kTile];
  __shared__ float ws[2][8];
  const Geo& G = A.geo;
  const int p = threadIdx.x;
  for (uint32_t LT = blockIdx.x; LT < G.n_ltiles; LT += gridDim.x) {
    const LTile lt = decode_ltile(A.ws, G.L, LT);
    float lm = 0.0f;
    if ((lt.start & 3) == 0) {
      // 16-byte aligned layer tile: 128-bit loads in the fixed lane order
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t off = 1024u * i + 4u * p;
        if (off >= lt.len) continue;
        const uint32_t nv = lt.len - off < 4u ? lt.len - off : 4u;
        const float4 mv = __ldcs(reinterpret_cast<const float4*>(A.m + lt.start + off));
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if ((uint32_t)c < nv) lm = __fadd_rn(lm, __fmul_rn(f4get(mv, c), f4get(mv, c)));
      }
    } else {
#pragma unroll 4
      for (int j = 0; j < 16; ++j) {
        const uint32_t idx = p + kThreads * j;
        float q = 0.0f;
        if (idx < lt.len) {
          const float mk = __ldcs(A.m + lt.start + idx);
          q = __fmul_rn(mk, mk);
        }
        sq[idx] = q;
      }
      __syncthreads();
      lm = lane_sum_sq(sq, p);
    }
    float tm, unused;
    block_sum2(lm, 0.0f, ws, tm, unused);
    if (p == 0) A.ws.lpart[LT] = tm;
    __syncthreads();
  }
}

// Pass 2, one warp per layer: rms_l = ||m_l|| / sqrt(n_l).
__global__ void __launch_bounds__(kThreads) k_lamb_begin_rms(const WarmupArgs A) {
  const Geo& G = A.geo;
  const int lane = threadIdx.x & 31;
  for (uint32_t l = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); l < G.L;
       l += gridDim.x * (kThreads / 32)) {
    const uint32_t b = __ldg(A.ws.ltile_pref + l);
    const uint32_t ntl = __ldg(A.ws.ltile_pref + l + 1) - b;
    const float nrm = __fsqrt_rn(ordered_sum(A.ws.lpart + b, ntl, lane));
    if (lane == 0) {
      const uint64_t nl = __ldg(A.ws.layer_off + l + 1) - __ldg(A.ws.layer_off + l);
      A.ws.rms[l] = __fdiv_rn(nrm, __fsqrt_rn(__ull2float_rn(nl)));
    }
  }
}

// Pass 3, one CTA: mean of the rms over layers (in layer order, from 0),
// s_l = mean / rms_l (1 if rms_l = 0), c_avg = c_sum / T_w, r = 1,
// c_prev = c_prev2 = c_avg.
__global__ void __launch_bounds__(kThreads) k_lamb_begin_final(const WarmupArgs A) {
  __shared__ float s_mean;
  const Geo& G = A.geo;
  if (threadIdx.x == 0) {
    float mean = 0.0f;
    for (uint32_t l = 0; l < G.L; ++l) mean = __fadd_rn(mean, A.ws.rms[l]);
    s_mean = __fdiv_rn(mean, (float)G.L);
  }
  __syncthreads();
  const float fT = (float)A.warmup_steps;
  for (uint32_t l = threadIdx.x; l < G.L; l += kThreads) {
    const float rms = A.ws.rms[l];
    A.ls.s[l] = rms == 0.0f ? 1.0f : __fdiv_rn(s_mean, rms);
    const float ca = __fdiv_rn(A.ls.c_sum[l], fT);
    A.ls.c_avg[l] = ca;
    A.ls.r_prev[l] = 1.0f;
    A.ls.c_prev[l] = ca;
    A.ls.c_prev2[l] = ca;
  }
}

}  // namespace

cudaError_t launch_warmup_adam(const WarmupArgs& a, bool bf16, int sms, cudaStream_t s) {
  const uint64_t nt = a.geo.n_tiles;
  if (bf16) k_warmup_adam<true><<<grid_for(k_warmup_adam<true>, sms, nt), kThreads, 0, s>>>(a);
  else k_warmup_adam<false><<<grid_for(k_warmup_adam<false>, sms, nt), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_warmup_lamb(const WarmupArgs& a, bool bf16, int sms, cudaStream_t s) {
  const uint64_t nlt = a.geo.n_ltiles;
  if (bf16) k_warmup_lamb_a<true><<<grid_for(k_warmup_lamb_a<true>, sms, nlt), kThreads, 0, s>>>(a);
  else k_warmup_lamb_a<false><<<grid_for(k_warmup_lamb_a<false>, sms, nlt), kThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const uint64_t lw = (a.geo.L + kThreads / 32 - 1) / (kThreads / 32);
  k_warmup_lamb_c<<<grid_for(k_warmup_lamb_c, sms, lw), kThreads, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_warmup_lamb_b<<<grid_for(k_warmup_lamb_b, sms, a.geo.n_tiles), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_lamb_begin(const WarmupArgs& a, int sms, cudaStream_t s) {
  k_lamb_begin_tiles<<<grid_for(k_lamb_begin_tiles, sms, a.geo.n_ltiles), kThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const uint64_t lw = (a.geo.L + kThreads / 32 - 1) / (kThreads / 32);
  k_lamb_begin_rms<<<grid_for(k_lamb_begin_rms, sms, lw), kThreads, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_lamb_begin_final<<<1, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ob
