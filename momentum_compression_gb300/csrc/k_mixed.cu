// Layerwise mixed bit widths ("1bit Adam" write-up, §3.2 table: a bit width
// and an update period per parameter type; §6 layerwise_bits [1, 2, 1, 16]).
// The layers of one width form a fused buffer of their own; this file holds
// the codecs of the widths other than 1:
//
//   b-bit (b = 2, 4, 8): the quantizer of the gradient quantization
//   tutorial ("FP32 → INT8 量化" and its GradientQuantizeINT8 example, which
//   takes the width as an argument) per block of 256 elements:
//   scale = max|x|/(2^(b-1)-1), stochastic rounding, clamp to
//   +-(2^(b-1)-1), with error feedback e' = x - q*scale.  Codes are packed b
//   bits per element, LSB first, two's complement.  The uniform of worker
//   w's element k is Philox word (w*n_pad + k)&3 of counter
//   ((w*n_pad + k)>>2, step); the server's use W*n_pad + k.
//
//   FP16: x rounded to IEEE binary16 (nearest, ties to even) with error
//   feedback, sent on every 10th step only; on the other steps the workers
//   keep x whole as their error, the server does not run, m = 0 and p is
//   left as it is.
//
// Kernels.  One warp per block of 256 elements (lane j holds elements
// 4j..4j+3 and 128+4j..128+4j+3): the worker kernel handles a block for all
// W workers in turn (m loaded once; the next worker's g and e are loaded
// while the current one is quantised); the server sums the W decoded
// messages in worker order; the update decodes the server message.  The
// FP16 kernels are elementwise, four elements per thread.
#include <cuda_fp16.h>

#include "ob_internal.cuh"
#include "philox.cuh"

namespace ob {
namespace {

constexpr int kWarps = kThreads / 32;

// Elements of this lane's half h that are real (k < n): 0..4.
__device__ __forceinline__ int valid4(uint64_t k, uint64_t n) {
  return k >= n ? 0 : (n - k >= 4 ? 4 : (int)(n - k));
}

// Code words of one lane-half: BITS*4 bits (4 fields); LPW lanes share a
// word.  Returns the word index inside the block and the bit offset of the
// lane's first field.
template <int BITS>
struct CodeSlot {
  static constexpr int kLPW = 8 / BITS;             // lanes per word
  static constexpr int kHalfWords = 4 * BITS;       // words per 128 elements
  static constexpr int kBlockWords = 8 * BITS;      // words per 256 elements
  static constexpr uint32_t kMask = (1u << BITS) - 1u;
  __device__ static int word(int h, int lane) { return h * kHalfWords + lane / kLPW; }
  __device__ static int shift(int lane) { return 4 * BITS * (lane % kLPW); }
};

// Signed field c (two's complement, BITS wide) of a code word already
// shifted to the lane's first field, as a float: the field is sign-extended
// by bfe.s32 and converted exactly through 1.5*2^23 (|q| < 2^22), which
// keeps the conversion on the integer and FMA pipes.
template <int BITS>
__device__ __forceinline__ float code_val(uint32_t v, int c) {
  int32_t q;
  asm("bfe.s32 %0, %1, %2, %3;" : "=r"(q) : "r"(v), "r"(BITS * c), "r"(BITS));
  return __fsub_rn(__int_as_float(0x4B400000 + q), 12582912.0f);
}

// Quantises the lane's 8 values of one block (x, nv real values per half)
// with error feedback; writes the code words (whole words, by the lanes
// that own them), the block scale and the residual e' (padding 0).
// The quantizer's Philox round keys are computed once on the host and
// passed to the kernels as a parameter: the rounds read them from the
// constant bank.  (Held in registers they took 20 of them, which the 3-CTA
// bound of the worker kernel could not spare; formed round by round, as the
// server did, they cost 20 additions per call.  Both forms measured about
// 4% slower.)
// PAIR: both halves' Philox outputs are drawn side by side (two independent
// chains; the server, 2% faster) or one at a time (the worker kernel, where
// the pair's registers spill at its 3-CTA bound: 23% slower).
template <int BITS, bool PAIR>
__device__ __forceinline__ void quantize_block(const float4 (&x)[2], const int (&nv)[2],
                                               uint64_t u_index0, uint64_t step,
                                               const PhiloxKeys& K, int lane,
                                               uint32_t* __restrict__ codes, float* scale_out,
                                               float4 (&e_out)[2]) {
  constexpr float qmax = (float)((1 << (BITS - 1)) - 1);
  using S = CodeSlot<BITS>;
  // fmaxf returns the other operand when one is NaN: a NaN never wins
  float mx = 0.0f;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (c < nv[h]) mx = fmaxf(mx, fabsf(f4get(x[h], c)));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
  const float scale = mx == 0.0f ? 0.0f : __fdiv_rn(mx, qmax);
  if (lane == 0) *scale_out = scale;
  // the halves' Philox counters (u_index0 + 128h + 4 lane is a multiple
  // of 4); the outputs are used only where a value is real and the scale
  // is not 0
  uint4 rnds[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint64_t grp = (u_index0 + 128 * h + 4 * lane) >> 2;
    rnds[h] = make_uint4((uint32_t)grp, (uint32_t)(grp >> 32), (uint32_t)step,
                         (uint32_t)(step >> 32));
  }
  if constexpr (PAIR) philox4x32_10_x2(rnds[0], rnds[1], K);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint4 rnd = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (PAIR) {
      rnd = rnds[h];
    } else if (nv[h] > 0 && scale != 0.0f) {
      rnd = philox4x32_10(rnds[h], K);
    }
    uint32_t piece = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float qf = 0.0f;
      if (c < nv[h] && scale != 0.0f) {
        const float xs = __fdiv_rn(f4get(x[h], c), scale);
        const float f = floorf(xs);
        const float fr = __fsub_rn(xs, f);
        qf = __fadd_rn(f, (uniform_of(word_of(rnd, c)) < fr) ? 1.0f : 0.0f);
        qf = qf > qmax ? qmax : qf;
        qf = qf < -qmax ? -qmax : qf;
        if (qf != qf) qf = 0.0f;
      }
      f4at(e_out[h], c) = c < nv[h] ? __fsub_rn(f4get(x[h], c), __fmul_rn(qf, scale)) : 0.0f;
      piece |= ((uint32_t)(int32_t)qf & S::kMask) << (BITS * c);
    }
    uint32_t w = piece << S::shift(lane);
#pragma unroll
    for (int o = 1; o < S::kLPW; o <<= 1) w |= __shfl_xor_sync(kFull, w, o);
    if (lane % S::kLPW == 0) codes[S::word(h, lane)] = w;
  }
}

// ---------------------------------------------------------------------------
// b-bit codec
// ---------------------------------------------------------------------------

template <bool BF16, int BITS>
__global__ void __launch_bounds__(kThreads, 3) k_qb_compress(const QbCompressArgs A,
                                                              const PhiloxKeys K) {
  const int lane = threadIdx.x & 31;
  const uint64_t nblk = A.n_pad / 256;
  const uint64_t warps = (uint64_t)gridDim.x * kWarps;
  const float ob1 = __fsub_rn(1.0f, A.b1);
  for (uint64_t b = (uint64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); b < nblk; b += warps) {
    int nv[2];
    float4 mv[2], gv[2], ev[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint64_t k = b * 256 + 128 * h + 4 * lane;
      nv[h] = valid4(k, A.n);
      mv[h] = __ldcs(reinterpret_cast<const float4*>(A.m + k));
      gv[h] = load_grad4<BF16>(A.g[0], k);
      ev[h] = __ldcs(reinterpret_cast<const float4*>(A.e[0] + k));
    }
    for (uint32_t w = 0; w < A.W; ++w) {
      // the next worker's loads are in flight while this one is quantised
      float4 gn[2], en[2];
      if (w + 1 < A.W) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint64_t k = b * 256 + 128 * h + 4 * lane;
          gn[h] = load_grad4<BF16>(A.g[w + 1], k);
          en[h] = __ldcs(reinterpret_cast<const float4*>(A.e[w + 1] + k));
        }
      }
      float4 x[2];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float mw = __fadd_rn(__fmul_rn(A.b1, f4get(mv[h], c)),
                                     __fmul_rn(ob1, f4get(gv[h], c)));
          float xv = __fadd_rn(mw, f4get(ev[h], c));
          if (A.clip > 0.0f) {
            xv = xv > A.clip ? A.clip : xv;
            xv = xv < -A.clip ? -A.clip : xv;
          }
          f4at(x[h], c) = c < nv[h] ? xv : 0.0f;
        }
      float4 r[2];
      quantize_block<BITS, false>(x, nv, (uint64_t)w * A.n_pad + b * 256, A.step, K, lane,
                           A.codes + (uint64_t)w * A.row_words + b * CodeSlot<BITS>::kBlockWords,
                           A.scales + (uint64_t)w * nblk + b, r);
#pragma unroll
      for (int h = 0; h < 2; ++h)
        __stcs(reinterpret_cast<float4*>(A.e[w] + b * 256 + 128 * h + 4 * lane), r[h]);
      if (w + 1 < A.W) {
        gv[0] = gn[0];
        gv[1] = gn[1];
        ev[0] = en[0];
        ev[1] = en[1];
      }
    }
  }
}

// 3 CTAs per SM (80 registers, no spill; unbounded it took 127 and ran 2):
// the 2-bit server 0.141 -> 0.129 ms on ResNet-50's group (0.123 ms with the round
// keys as a kernel parameter).
template <int BITS>
__global__ void __launch_bounds__(kThreads, 3) k_qb_server(const QbServerArgs A,
                                                           const PhiloxKeys K) {
  using S = CodeSlot<BITS>;
  const int lane = threadIdx.x & 31;
  const uint64_t nblk = A.n_pad / 256;
  const uint64_t warps = (uint64_t)gridDim.x * kWarps;
  const float fW = (float)A.W, inv_w = inv_workers(A.W);
  for (uint64_t b = (uint64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); b < nblk; b += warps) {
    int nv[2];
    float4 es[2], z[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint64_t k = b * 256 + 128 * h + 4 * lane;
      nv[h] = valid4(k, A.n);
      es[h] = __ldcs(reinterpret_cast<const float4*>(A.e_s + k));
      z[h] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const uint32_t* cb = A.codes + b * S::kBlockWords;
    // workers in batches of 8: all of a batch's words and scales are loaded
    // before they are added, in worker order
    for (uint32_t w0 = 0; w0 < A.W; w0 += 8) {
      uint32_t wd[8][2];
      float sc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (w0 + i < A.W) {
          const uint32_t* row = cb + (uint64_t)(w0 + i) * A.row_words;
          wd[i][0] = __ldcs(row + S::word(0, lane));
          wd[i][1] = __ldcs(row + S::word(1, lane));
          sc[i] = __ldcs(A.scales + (uint64_t)(w0 + i) * nblk + b);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (w0 + i < A.W) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t v = wd[i][h] >> S::shift(lane);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              f4at(z[h], c) = __fadd_rn(f4get(z[h], c), __fmul_rn(code_val<BITS>(v, c), sc[i]));
          }
        }
      }
    }
    float4 y[2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        f4at(y[h], c) =
            c < nv[h] ? __fadd_rn(f4get(es[h], c), div_by_workers(f4get(z[h], c), fW, inv_w))
                      : 0.0f;
    float4 r[2];
    quantize_block<BITS, true>(y, nv, (uint64_t)A.W * A.n_pad + b * 256, A.step, K, lane,
                         A.scodes + b * S::kBlockWords, A.sscales + b, r);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      __stcs(reinterpret_cast<float4*>(A.e_s + b * 256 + 128 * h + 4 * lane), r[h]);
  }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) k_qb_adam(const QbUpdateArgs A) {
  using S = CodeSlot<BITS>;
  const int lane = threadIdx.x & 31;
  const uint64_t nblk = A.n_pad / 256;
  const uint64_t warps = (uint64_t)gridDim.x * kWarps;
  for (uint64_t b = (uint64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); b < nblk; b += warps) {
    const float sc = __ldcs(A.sscales + b);
    uint32_t wd[2];
    float4 vv[2], pv[2];
    int nv[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint64_t k = b * 256 + 128 * h + 4 * lane;
      nv[h] = valid4(k, A.n);
      wd[h] = __ldcs(A.scodes + b * S::kBlockWords + S::word(h, lane));
      vv[h] = __ldcs(reinterpret_cast<const float4*>(A.v + k));
      pv[h] = __ldcs(reinterpret_cast<const float4*>(A.p + k));
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint64_t k = b * 256 + 128 * h + 4 * lane;
      float4 mv;
      const uint32_t v = wd[h] >> S::shift(lane);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (c < nv[h]) {
          const float mk = __fmul_rn(code_val<BITS>(v, c), sc);
          const float u = __fdiv_rn(mk, __fadd_rn(__fsqrt_rn(f4get(vv[h], c)), A.eps));
          f4at(pv[h], c) = __fsub_rn(f4get(pv[h], c), __fmul_rn(A.lr, u));
          f4at(mv, c) = mk;
        } else {
          f4at(mv, c) = 0.0f;
        }
      }
      __stcs(reinterpret_cast<float4*>(A.m + k), mv);
      if (nv[h] == 4) {
        __stcs(reinterpret_cast<float4*>(A.p + k), pv[h]);
      } else {
#pragma unroll
        for (int c = 0; c < 3; ++c)
          if (c < nv[h]) A.p[k + c] = f4get(pv[h], c);  // padding of p is never written
      }
    }
  }
}

// ---------------------------------------------------------------------------
// FP16 codec
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  return (uint32_t)__half_as_ushort(__float2half_rn(a)) |
         ((uint32_t)__half_as_ushort(__float2half_rn(b)) << 16);
}

__device__ __forceinline__ float half_lo(uint32_t u) {
  return __half2float(__ushort_as_half((unsigned short)(u & 0xffffu)));
}

__device__ __forceinline__ float half_hi(uint32_t u) {
  return __half2float(__ushort_as_half((unsigned short)(u >> 16)));
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads) k_f16_compress(const F16Args A) {
  const uint64_t groups = A.n_pad / 4;
  const float ob1 = __fsub_rn(1.0f, A.b1);
  for (uint64_t i = (uint64_t)blockIdx.x * kThreads + threadIdx.x; i < groups;
       i += (uint64_t)gridDim.x * kThreads) {
    const uint64_t k = 4 * i;
    const int nv = valid4(k, A.n);
    const float4 mv = __ldcs(reinterpret_cast<const float4*>(A.m + k));
    for (uint32_t w = 0; w < A.W; ++w) {
      const float4 gv = load_grad4<BF16>(A.g[w], k);
      const float4 ev = __ldcs(reinterpret_cast<const float4*>(A.e[w] + k));
      float4 x, r;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float mw = __fadd_rn(__fmul_rn(A.b1, f4get(mv, c)), __fmul_rn(ob1, f4get(gv, c)));
        float xv = __fadd_rn(mw, f4get(ev, c));
        if (A.clip > 0.0f) {
          xv = xv > A.clip ? A.clip : xv;
          xv = xv < -A.clip ? -A.clip : xv;
        }
        f4at(x, c) = c < nv ? xv : 0.0f;
      }
      if (A.send) {
        const uint2 hv = make_uint2(pack_half2(x.x, x.y), pack_half2(x.z, x.w));
        r = make_float4(__fsub_rn(x.x, half_lo(hv.x)), __fsub_rn(x.y, half_hi(hv.x)),
                        __fsub_rn(x.z, half_lo(hv.y)), __fsub_rn(x.w, half_hi(hv.y)));
        __stcs(reinterpret_cast<uint2*>(A.h + (uint64_t)w * A.n_pad + k), hv);
      } else {
        r = x;
      }
      __stcs(reinterpret_cast<float4*>(A.e[w] + k), r);
    }
  }
}

__global__ void __launch_bounds__(kThreads) k_f16_server(const F16Args A) {
  const uint64_t groups = A.n_pad / 4;
  const float fW = (float)A.W, inv_w = inv_workers(A.W);
  for (uint64_t i = (uint64_t)blockIdx.x * kThreads + threadIdx.x; i < groups;
       i += (uint64_t)gridDim.x * kThreads) {
    const uint64_t k = 4 * i;
    const int nv = valid4(k, A.n);
    float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (uint32_t w = 0; w < A.W; ++w) {
      const uint2 hv = __ldcs(reinterpret_cast<const uint2*>(A.h + (uint64_t)w * A.n_pad + k));
      z.x = __fadd_rn(z.x, half_lo(hv.x));
      z.y = __fadd_rn(z.y, half_hi(hv.x));
      z.z = __fadd_rn(z.z, half_lo(hv.y));
      z.w = __fadd_rn(z.w, half_hi(hv.y));
    }
    const float4 es = __ldcs(reinterpret_cast<const float4*>(A.e_s + k));
    float4 y;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      f4at(y, c) = c < nv ? __fadd_rn(f4get(es, c), div_by_workers(f4get(z, c), fW, inv_w))
                          : 0.0f;
    const uint2 hs = make_uint2(pack_half2(y.x, y.y), pack_half2(y.z, y.w));
    const float4 r = make_float4(__fsub_rn(y.x, half_lo(hs.x)), __fsub_rn(y.y, half_hi(hs.x)),
                                 __fsub_rn(y.z, half_lo(hs.y)), __fsub_rn(y.w, half_hi(hs.y)));
    __stcs(reinterpret_cast<uint2*>(A.hs + k), hs);
    __stcs(reinterpret_cast<float4*>(A.e_s + k), r);
  }
}

__global__ void __launch_bounds__(kThreads) k_f16_adam(const F16Args A) {
  const uint64_t groups = A.n_pad / 4;
  for (uint64_t i = (uint64_t)blockIdx.x * kThreads + threadIdx.x; i < groups;
       i += (uint64_t)gridDim.x * kThreads) {
    const uint64_t k = 4 * i;
    const int nv = A.send ? valid4(k, A.n) : 0;
    float4 mv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (nv > 0) {
      const uint2 hv = __ldcs(reinterpret_cast<const uint2*>(A.hs + k));
      const float4 vv = __ldcs(reinterpret_cast<const float4*>(A.v + k));
      float4 pv = __ldcs(reinterpret_cast<const float4*>(A.p + k));
      const float hm[4] = {half_lo(hv.x), half_hi(hv.x), half_lo(hv.y), half_hi(hv.y)};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (c < nv) {
          const float u = __fdiv_rn(hm[c], __fadd_rn(__fsqrt_rn(f4get(vv, c)), A.eps));
          f4at(pv, c) = __fsub_rn(f4get(pv, c), __fmul_rn(A.lr, u));
          f4at(mv, c) = hm[c];
        }
      }
      if (nv == 4) {
        __stcs(reinterpret_cast<float4*>(A.p + k), pv);
      } else {
#pragma unroll
        for (int c = 0; c < 3; ++c)
          if (c < nv) A.p[k + c] = f4get(pv, c);
      }
    }
    __stcs(reinterpret_cast<float4*>(A.m + k), mv);
  }
}

uint64_t warp_ctas(uint64_t n_pad) {
  return (n_pad / 256 + kWarps - 1) / kWarps;
}

}  // namespace

cudaError_t launch_qb_compress(const QbCompressArgs& a, int bits, bool bf16, int sms,
                               cudaStream_t s) {
  const uint64_t ctas = warp_ctas(a.n_pad);
  const PhiloxKeys K = philox_keys((uint32_t)a.seed, (uint32_t)(a.seed >> 32));
#define OB_QB_COMPRESS(BF, B)                                                         \
  k_qb_compress<BF, B><<<grid_for(k_qb_compress<BF, B>, sms, ctas), kThreads, 0, s>>>(a, K)
  if (bf16) {
    if (bits == 2) OB_QB_COMPRESS(true, 2);
    else if (bits == 4) OB_QB_COMPRESS(true, 4);
    else OB_QB_COMPRESS(true, 8);
  } else {
    if (bits == 2) OB_QB_COMPRESS(false, 2);
    else if (bits == 4) OB_QB_COMPRESS(false, 4);
    else OB_QB_COMPRESS(false, 8);
  }
#undef OB_QB_COMPRESS
  return cudaGetLastError();
}

template <int B>
void run_qb_server(const QbServerArgs& a, int sms, uint64_t ctas, cudaStream_t s) {
  const PhiloxKeys K = philox_keys((uint32_t)a.seed, (uint32_t)(a.seed >> 32));
  k_qb_server<B><<<grid_for(k_qb_server<B>, sms, ctas), kThreads, 0, s>>>(a, K);
}

cudaError_t launch_qb_server(const QbServerArgs& a, int bits, int sms, cudaStream_t s) {
  const uint64_t ctas = warp_ctas(a.n_pad);
  if (bits == 2) run_qb_server<2>(a, sms, ctas, s);
  else if (bits == 4) run_qb_server<4>(a, sms, ctas, s);
  else run_qb_server<8>(a, sms, ctas, s);
  return cudaGetLastError();
}

cudaError_t launch_qb_adam(const QbUpdateArgs& a, int bits, int sms, cudaStream_t s) {
  const uint64_t ctas = warp_ctas(a.n_pad);
  if (bits == 2) k_qb_adam<2><<<grid_for(k_qb_adam<2>, sms, ctas), kThreads, 0, s>>>(a);
  else if (bits == 4) k_qb_adam<4><<<grid_for(k_qb_adam<4>, sms, ctas), kThreads, 0, s>>>(a);
  else k_qb_adam<8><<<grid_for(k_qb_adam<8>, sms, ctas), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_f16_compress(const F16Args& a, bool bf16, int sms, cudaStream_t s) {
  const uint64_t ctas = (a.n_pad / 4 + kThreads - 1) / kThreads;
  if (bf16) k_f16_compress<true><<<grid_for(k_f16_compress<true>, sms, ctas), kThreads, 0, s>>>(a);
  else k_f16_compress<false><<<grid_for(k_f16_compress<false>, sms, ctas), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_f16_server(const F16Args& a, int sms, cudaStream_t s) {
  const uint64_t ctas = (a.n_pad / 4 + kThreads - 1) / kThreads;
  k_f16_server<<<grid_for(k_f16_server, sms, ctas), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_f16_adam(const F16Args& a, int sms, cudaStream_t s) {
  const uint64_t ctas = (a.n_pad / 4 + kThreads - 1) / kThreads;
  k_f16_adam<<<grid_for(k_f16_adam, sms, ctas), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ob
