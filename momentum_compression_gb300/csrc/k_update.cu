// Unpack + update kernels of the 1-bit compressed optimizer step, and the
// standalone decompression and error materialisation.
//
//   1-bit Adam (1-bit LAMB summary, paragraph 1: the frozen denominator
//   sqrt(v_Tw); "1bit Adam" write-up, 2.1):
//     m = sscale*sign(sbit);  p = p - lr*(m/(sqrt(v_Tw)+eps))
//   1-bit LAMB (1-bit LAMB summary, paragraphs 1-3), pass A:
//     m_t = sscale*sign/sigma_l; g = (m_t - b1*m_{t-1})/(1-b1)
//     v_t = b2*v_t + (1-b2)*g^2;  R_l = max over the layer of v_Tw/v_t
//   then per layer (by the last CTA of pass A):
//     r = clip(clip(R_l, (1-r_thr)r_prev, (1+r_thr)r_prev), r_min, r_max)
//     c = clip(c_avg*r, c_min, c_max); c_prev2 <- c_prev <- c; r_prev <- r
//   pass B:
//     p = p - (lr*c_l)*(m_t/(sqrt(v_Tw)+eps))
// All operations are rounded one by one (no contraction), with IEEE
// division and square root.
#include <type_traits>

#include "ob_internal.cuh"
#include "ptx.cuh"

namespace ob {
namespace {

// Thread 0 asks the copy engine to bring tile Tn's rows of the given fp32
// arrays and the runs of the given sign-word arrays covering it into L2,
// while the CTA works on the current tile: the next grid-stride tile's
// loads then hit L2.  Tiles start on multiples of 32 elements and hold a
// multiple of 32, so the rows are 128-byte aligned; the word runs are
// widened to 16-byte boundaries, which stay inside the rows (padded to 16
// bytes).  Null arrays are skipped.
__device__ __forceinline__ void prefetch_tile(const Geo& G, uint32_t Tn, const float* a0,
                                              const float* a1, const float* a2,
                                              const uint32_t* w0, const uint32_t* w1) {
  if (threadIdx.x != 0 || Tn >= G.n_tiles) return;
  const Tile t = decode_tile(G, Tn);
  const uint32_t bytes = t.len * 4u;
  if (a0) bulk_prefetch_l2(a0 + t.start, bytes);
  if (a1) bulk_prefetch_l2(a1 + t.start, bytes);
  if (a2) bulk_prefetch_l2(a2 + t.start, bytes);
  const uint64_t wb = (t.start >> 5) & ~3ull;
  const uint64_t we = (((t.start + t.len + 31) >> 5) + 3) & ~3ull;
  if (w0) bulk_prefetch_l2(w0 + wb, (uint32_t)(we - wb) * 4u);
  if (w1) bulk_prefetch_l2(w1 + wb, (uint32_t)(we - wb) * 4u);
}

__global__ void __launch_bounds__(kThreads) k_adam_update(const UpdateArgs A) {
  const Geo& G = A.geo;
  const int p = threadIdx.x;
  const float* __restrict__ vf = A.v_frozen;
  float* __restrict__ pp = A.p;
  float* __restrict__ mm = A.m;
  for (uint32_t T = blockIdx.x; T < G.n_tiles; T += gridDim.x) {
    // (no L2 prefetch of the next tile here: it gained 2% at 1e8 elements
    // and lost 25% at 1.3e9; plain loads and stores: with the streaming
    // .cs hints the kernel measured 4.6% slower at 1.3e9 elements)
    const Tile tl = decode_tile(G, T);
    const float osc = __ldcg(A.sscales + tl.g);
    // all loads of the tile first (4 sign words, 4 x 2 128-bit rows), then
    // the arithmetic, then the stores
    uint32_t wd[4];
    float4 vv[4], pv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t off = 1024u * i + 4u * p;
      const uint64_t k0 = tl.start + off;
      const bool live = off < tl.len && k0 < G.n;
      wd[i] = live ? __ldg(A.sbits + (k0 >> 5)) >> (4 * (p & 7)) : 0u;
      vv[i] = live ? __ldg(reinterpret_cast<const float4*>(vf + k0)) : make_float4(0.f, 0.f, 0.f, 0.f);
      pv[i] = live ? *reinterpret_cast<const float4*>(pp + k0) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t off = 1024u * i + 4u * p;
      if (off >= tl.len) continue;
      const uint64_t k0 = tl.start + off;
      float4 mo;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (k0 + c < G.n) {
          const float mk = signed_by_bit(osc, wd[i], c);
          const float d = __fadd_rn(__fsqrt_rn(f4get(vv[i], c)), A.eps);
          const float u = __fdiv_rn(mk, d);
          f4at(pv[i], c) = __fsub_rn(f4get(pv[i], c), __fmul_rn(A.lr, u));
          f4at(mo, c) = mk;
        } else {
          f4at(mo, c) = 0.0f;  // padding: m = 0, p untouched
        }
      }
      if (mm) *reinterpret_cast<float4*>(mm + k0) = mo;  // m == null: kept as signs
      if (k0 < G.n) *reinterpret_cast<float4*>(pp + k0) = pv[i];
    }
  }
}

// Per-layer ratio and coefficient, run by one CTA.
__device__ void lamb_ratio_all(const UpdateArgs& A) {
  const LambHP& h = A.hp;
  for (uint32_t l = threadIdx.x; l < A.geo.L; l += kThreads) {
    const float R = __uint_as_float(__ldcg(A.ws.Rbits + l));
    const float rp = A.ls.r_prev[l];
    float r;
    if (h.frozen) {
      r = 1.0f;
    } else {
      const float lo = __fmul_rn(__fsub_rn(1.0f, h.r_thr), rp);
      const float hi = __fmul_rn(__fadd_rn(1.0f, h.r_thr), rp);
      r = fmin_plain(fmax_plain(R, lo), hi);
      r = fmin_plain(fmax_plain(r, h.r_min), h.r_max);
    }
    float c = __fmul_rn(A.ls.c_avg[l], r);
    c = fmin_plain(fmax_plain(c, h.c_min), h.c_max);
    A.ls.c_prev2[l] = A.ls.c_prev[l];
    A.ls.c_prev[l] = c;
    A.ls.r_prev[l] = r;
    A.ls.c_t[l] = c;
    A.ws.Rbits[l] = 0u;
  }
}

// SIGNM: the momentum is held in sign form -- m_{t-1} = sscale_prev *
// sign(sbit_prev)/sigma_l from the previous step's server output (double
// buffered by the caller) instead of a dense buffer, and m_t is not written
// (it is the current server output over sigma_l).
// Sign form at 4 CTAs per SM (64 registers, no spill): 32 warps overlap
// the loads better (BERT-large passes A + B 1.44 -> 1.38 ms); the dense
// form keeps 3.
template <bool SIGNM>
__global__ void __launch_bounds__(kThreads, SIGNM ? 4 : 3) k_lamb_pass_a(const UpdateArgs A) {
  __shared__ int s_last;
  const Geo& G = A.geo;
  const int p = threadIdx.x;
  // Running max of the ratio for layer l, kept across this CTA's tiles and
  // flushed with atomicMax only when the layer changes (and at the end):
  // one atomic per warp and layer, instead of per tile -- with one large
  // layer, per-tile atomics on the same word serialised the whole pass.
  uint32_t l = ~0u;
  float rmax = 0.0f;
  // one atomic per warp when all its lanes are in the same layer, else one
  // per lane (rmax > 0 only after a real ratio, so l is a layer then)
  auto flush = [&]() {
    const uint32_t l0 = __shfl_sync(kFull, l, 0);
    if (__all_sync(kFull, l == l0)) {
      float wmax = rmax;
      for (int o = 16; o >= 1; o >>= 1) wmax = fmax_plain(wmax, __shfl_xor_sync(kFull, wmax, o));
      if ((p & 31) == 0 && wmax > 0.0f) atomicMax(A.ws.Rbits + l, __float_as_uint(wmax));
    } else if (rmax > 0.0f) {
      atomicMax(A.ws.Rbits + l, __float_as_uint(rmax));
    }
  };
  for (uint32_t T = blockIdx.x; T < G.n_tiles; T += gridDim.x) {
    const Tile tl = decode_tile(G, T);
    const float osc = __ldcg(A.sscales + tl.g);
    [[maybe_unused]] const float oscp = SIGNM ? __ldcg(A.sscales_prev + tl.g) : 0.0f;
    const uint32_t l_t = __ldg(A.ws.tile_layer + T);
    const uint64_t lend_t = __ldg(A.ws.layer_off + l_t + 1);
    const float s_t = __ldg(A.ls.s + l_t);
    // all loads of the tile first
    uint32_t wd[4];
    [[maybe_unused]] uint32_t wdp[4];
    float4 mv[4], vt[4], vf[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t off = 1024u * i + 4u * p;
      const uint64_t k0 = tl.start + off;
      const bool live = off < tl.len && k0 < G.n;
      const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
      wd[i] = live ? __ldg(A.sbits + (k0 >> 5)) >> (4 * (p & 7)) : 0u;
      if constexpr (SIGNM) {
        wdp[i] = live ? __ldg(A.sbits_prev + (k0 >> 5)) >> (4 * (p & 7)) : 0u;
      } else {
        mv[i] = live ? __ldcs(reinterpret_cast<const float4*>(A.m + k0)) : z4;
      }
      vt[i] = live ? __ldcs(reinterpret_cast<const float4*>(A.v_fresh + k0)) : z4;
      vf[i] = live ? __ldcs(reinterpret_cast<const float4*>(A.v_frozen + k0)) : z4;
    }
    // UNI: the whole tile lies in one layer; else the layers are walked
    // element by element and each layer's running max is flushed when the
    // walk leaves it
    if (__any_sync(kFull, l != l_t)) {
      flush();
      l = l_t;
      rmax = 0.0f;
    }
    auto body = [&](auto uni_tag) {
      constexpr bool UNI = decltype(uni_tag)::value;
      uint64_t lend = lend_t;
      // M/sigma = +-(sscale/sigma) exactly (IEEE division is symmetric in
      // sign): one division per layer instead of one per element
      float q_l = __fdiv_rn(osc, s_t);
      [[maybe_unused]] float qp_l = SIGNM ? __fdiv_rn(oscp, s_t) : 0.0f;
      // (With the momentum in sign form g takes only +-g_same and +-g_diff
      // per layer, but precomputing them measured slower: the per-element
      // division keeps the tile's loads overlapped with more work.)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint64_t k0 = tl.start + 1024u * i + 4u * p;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint64_t k = k0 + c;
          if (1024u * i + 4u * p >= tl.len || k >= G.n) {
            if constexpr (!SIGNM) f4at(mv[i], c) = 0.0f;
            continue;
          }
          if constexpr (!UNI) {
            const uint32_t l_old = l;
            if (advance_layer(A.ws.layer_off, G.L, k, l, lend)) {
              if (rmax > 0.0f) atomicMax(A.ws.Rbits + l_old, __float_as_uint(rmax));
              rmax = 0.0f;
              const float sg = __ldg(A.ls.s + l);
              q_l = __fdiv_rn(osc, sg);
              if constexpr (SIGNM) qp_l = __fdiv_rn(oscp, sg);
            }
          }
          const float mt = ((wd[i] >> c) & 1u) ? q_l : -q_l;
          float mprev;
          if constexpr (SIGNM) mprev = ((wdp[i] >> c) & 1u) ? qp_l : -qp_l;
          else mprev = f4get(mv[i], c);
          const float gt = __fdiv_rn(__fsub_rn(mt, __fmul_rn(A.b1, mprev)), A.ob1);
          const float v = __fadd_rn(__fmul_rn(A.b2, f4get(vt[i], c)),
                                    __fmul_rn(A.ob2, __fmul_rn(gt, gt)));
          if constexpr (!SIGNM) f4at(mv[i], c) = mt;
          f4at(vt[i], c) = v;
          const float ratio = __fdiv_rn(f4get(vf[i], c), v);
          if (ratio > rmax) rmax = ratio;  // NaN never wins
        }
      }
    };
    if (tl.start + tl.len <= lend_t || G.n <= lend_t) body(std::true_type{});
    else body(std::false_type{});
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t off = 1024u * i + 4u * p;
      if (off >= tl.len) continue;
      const uint64_t k0 = tl.start + off;
      if constexpr (!SIGNM) __stcs(reinterpret_cast<float4*>(A.m + k0), mv[i]);
      if (k0 < G.n) __stcs(reinterpret_cast<float4*>(A.v_fresh + k0), vt[i]);
    }
  }
  flush();
  // Last CTA of the grid: per-layer ratio and coefficient.
  __threadfence();
  __syncthreads();
  if (p == 0) {
    unsigned prev = atomicAdd(A.ws.gcnt + 0, 1u);
    s_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    lamb_ratio_all(A);
    if (p == 0) A.ws.gcnt[0] = 0u;
  }
}

// SIGNM: m_t = sscale*sign(sbit)/sigma_l from the server output (the
// momentum held in sign form) instead of a dense buffer.
template <bool SIGNM>
__global__ void __launch_bounds__(kThreads) k_lamb_pass_b(const UpdateArgs A) {
  const Geo& G = A.geo;
  const int p = threadIdx.x;
  for (uint32_t T = blockIdx.x; T < G.n_tiles; T += gridDim.x) {
    prefetch_tile(G, T + gridDim.x, A.v_frozen, A.p, SIGNM ? nullptr : A.m,
                  SIGNM ? A.sbits : nullptr, nullptr);
    const Tile tl = decode_tile(G, T);
    if (tl.start >= G.n) continue;
    const uint32_t l_t = __ldg(A.ws.tile_layer + T);
    const uint64_t lend_t = __ldg(A.ws.layer_off + l_t + 1);
    const float t1_t = __fmul_rn(A.lr, __ldcg(A.ls.c_t + l_t));
    [[maybe_unused]] const float osc = SIGNM ? __ldcg(A.sscales + tl.g) : 0.0f;
    [[maybe_unused]] uint32_t wd[4];
    float4 mv[4], vf[4], pv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t off = 1024u * i + 4u * p;
      const uint64_t k0 = tl.start + off;
      const bool live = off < tl.len && k0 < G.n;
      const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
      if constexpr (SIGNM)
        wd[i] = live ? __ldg(A.sbits + (k0 >> 5)) >> (4 * (p & 7)) : 0u;
      else
        mv[i] = live ? __ldcs(reinterpret_cast<const float4*>(A.m + k0)) : z4;
      vf[i] = live ? __ldcs(reinterpret_cast<const float4*>(A.v_frozen + k0)) : z4;
      pv[i] = live ? __ldcs(reinterpret_cast<const float4*>(A.p + k0)) : z4;
    }
    auto body = [&](auto uni_tag) {
      constexpr bool UNI = decltype(uni_tag)::value;
      uint32_t l = l_t;
      uint64_t lend = lend_t;
      float t1 = t1_t;
      // m_t = +-(sscale/sigma_l), the value pass A computed
      [[maybe_unused]] float q_l = SIGNM ? __fdiv_rn(osc, __ldg(A.ls.s + l_t)) : 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint64_t k0 = tl.start + 1024u * i + 4u * p;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint64_t k = k0 + c;
          if (1024u * i + 4u * p >= tl.len || k >= G.n) continue;
          if constexpr (!UNI) {
            if (advance_layer(A.ws.layer_off, G.L, k, l, lend)) {
              t1 = __fmul_rn(A.lr, __ldcg(A.ls.c_t + l));
              if constexpr (SIGNM) q_l = __fdiv_rn(osc, __ldg(A.ls.s + l));
            }
          }
          float mt;
          if constexpr (SIGNM) mt = ((wd[i] >> c) & 1u) ? q_l : -q_l;
          else mt = f4get(mv[i], c);
          const float d = __fadd_rn(__fsqrt_rn(f4get(vf[i], c)), A.eps);
          const float u = __fdiv_rn(mt, d);
          f4at(pv[i], c) = __fsub_rn(f4get(pv[i], c), __fmul_rn(t1, u));
        }
      }
    };
    if (tl.start + tl.len <= lend_t || G.n <= lend_t) body(std::true_type{});
    else body(std::false_type{});
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t off = 1024u * i + 4u * p;
      const uint64_t k0 = tl.start + off;
      if (off < tl.len && k0 < G.n) __stcs(reinterpret_cast<float4*>(A.p + k0), pv[i]);
    }
  }
}

template <bool LAYERED>
__global__ void __launch_bounds__(kThreads) k_decompress(const UpdateArgs A) {
  const Geo& G = A.geo;
  const int p = threadIdx.x;
  for (uint32_t T = blockIdx.x; T < G.n_tiles; T += gridDim.x) {
    const Tile tl = decode_tile(G, T);
    const float osc = __ldcg(A.sscales + tl.g);
    uint32_t l = 0;
    uint64_t lend = 0;
    // the magnitude of every value of the layer: sscale, or sscale/sigma_l
    // (+-sscale/sigma = (+-sscale)/sigma exactly: IEEE division is
    // symmetric in sign)
    float q_l = osc;
    if constexpr (LAYERED) {
      l = __ldg(A.ws.tile_layer + T);
      lend = __ldg(A.ws.layer_off + l + 1);
      q_l = __fdiv_rn(osc, __ldg(A.ls.s + l));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t off = 1024u * i + 4u * p;
      if (off >= tl.len) continue;
      const uint64_t k0 = tl.start + off;
      const uint32_t wd = __ldg(A.sbits + (k0 >> 5)) >> (4 * (p & 7));
      float4 o;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint64_t k = k0 + c;
        float M = 0.0f;
        if (k < G.n) {
          if constexpr (LAYERED) {
            if (advance_layer(A.ws.layer_off, G.L, k, l, lend))
              q_l = __fdiv_rn(osc, __ldg(A.ls.s + l));
          }
          M = ((wd >> c) & 1u) ? q_l : -q_l;
        }
        f4at(o, c) = M;
      }
      __stcs(reinterpret_cast<float4*>(A.out + k0), o);
    }
  }
}

// RESET = false: e := e - scale*sign (the deferred error made explicit).
// RESET = true:  e := scale*sign, so that the next decode gives exactly 0
//                (the periodic reset of the "1bit Adam" write-up, 4.1).
template <bool RESET>
__global__ void __launch_bounds__(kThreads) k_materialize(const MaterializeArgs A) {
  const Geo& G = A.geo;
  const int p = threadIdx.x;
  const uint32_t NW = A.nw;
  for (uint32_t T = A.T0 + blockIdx.x; T < A.T1; T += gridDim.x) {
    const Tile tl = decode_tile(G, T);
    if (tl.start >= G.n) continue;
    for (uint32_t w = 0; w <= NW; ++w) {
      // w < nw: worker errors; w == nw: the server error (if given)
      if (w == NW && !A.e_s) break;
      const uint64_t base = w < NW ? 0 : A.base;
      float* e = w < NW ? A.e[w] : A.e_s;
      const uint32_t* bw = w < NW ? A.bits + (uint64_t)w * G.words : A.sbits;
      const float sc = w < NW ? __ldcg(A.scales + (uint64_t)w * G.nc + tl.g)
                              : __ldcg(A.sscales + (tl.g - A.g0));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t off = 1024u * i + 4u * p;
        if (off >= tl.len) continue;
        const uint64_t k0 = tl.start + off;
        if (k0 >= G.n) continue;
        const uint64_t kl = k0 - base;  // base is a multiple of 32: same bit in the word
        const uint32_t wd = bw[kl >> 5] >> (4 * (p & 7));
        float4 ev = *reinterpret_cast<const float4*>(e + kl);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (k0 + c >= G.n) continue;
          const float so = ((wd >> c) & 1u) ? sc : -sc;
          f4at(ev, c) = RESET ? so : __fsub_rn(f4at(ev, c), so);
        }
        *reinterpret_cast<float4*>(e + kl) = ev;
      }
    }
  }
}

}  // namespace

cudaError_t launch_adam_update(const UpdateArgs& a, int sms, cudaStream_t s) {
  k_adam_update<<<grid_for(k_adam_update, sms, a.geo.n_tiles), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_lamb_pass_a(const UpdateArgs& a, int sms, cudaStream_t s) {
  if (a.m)
    k_lamb_pass_a<false><<<grid_for(k_lamb_pass_a<false>, sms, a.geo.n_tiles), kThreads, 0, s>>>(a);
  else
    k_lamb_pass_a<true><<<grid_for(k_lamb_pass_a<true>, sms, a.geo.n_tiles), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_lamb_pass_b(const UpdateArgs& a, int sms, cudaStream_t s) {
  if (a.m)
    k_lamb_pass_b<false><<<grid_for(k_lamb_pass_b<false>, sms, a.geo.n_tiles), kThreads, 0, s>>>(a);
  else
    k_lamb_pass_b<true><<<grid_for(k_lamb_pass_b<true>, sms, a.geo.n_tiles), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decompress(const UpdateArgs& a, bool layered, int sms,
                              cudaStream_t s) {
  if (layered)
    k_decompress<true><<<grid_for(k_decompress<true>, sms, a.geo.n_tiles), kThreads, 0, s>>>(a);
  else
    k_decompress<false><<<grid_for(k_decompress<false>, sms, a.geo.n_tiles), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_materialize(const MaterializeArgs& a, int sms, cudaStream_t s) {
  k_materialize<false><<<grid_for(k_materialize<false>, sms, a.T1 - a.T0), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_reset_errors(const MaterializeArgs& a, int sms, cudaStream_t s) {
  k_materialize<true><<<grid_for(k_materialize<true>, sms, a.T1 - a.T0), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ob
