// Stochastic rounding of a block-scaled value to a signed code (the
// gradient quantization tutorial, "FP32 → INT8 量化" and its
// GradientQuantizeINT8 example, which takes the width as an argument):
// x = g/scale correctly rounded, f = floor(x), q = f + (u < x - f), clamped
// to +-qmax, a NaN coding as 0; scale = max|g| / qmax over the block, u in
// [0, 1) on the 2^-24 grid.  Used by the INT8 quantizer (qmax = 127); the
// bound below holds for any qmax <= 127.  (The b-bit codec's kernels keep
// the division: there it is a small share of the work, and the fast path's
// registers measured slower.)
//
// code_exact computes the definition.  code_fast takes the quotient from
// the block's correctly rounded reciprocal instead of a division and tells
// whether its code is certainly the definition's:
//
// The code is ceil(x - u) (clamped) for every quotient x: x = f + fr with
// f = floor(x); fr > u gives f + 1 and fr <= u gives f, which is
// ceil(x - u) -- exactly so where fr = x - f is exact (x >= 0 or x <= -1,
// Sterbenz), and for x in (-1, 0), where fr = RN(1 + x), as long as 1 + x
// is more than 2^-25 (half an ulp below 1) from u.  With a normal block
// scale s (s >= 2^-126) and r = 1/s correctly rounded, y = RN(g*r) and
// x = RN(g/s) of a value of the block (|g| <= max|g| = qmax*s*(1 +- 2^-24),
// so |g/s| < 127.0001) differ by less than
// |g/s|*(2^-23 + 2^-48) + 2^-150 + ulp(x)/2 < 5*2^-18 (r and y each carry
// one rounding of relative size 2^-24, or an absolute 2^-150 below the
// normal range), and t = RN(y - u) lies within 2^-18 more of y - u.  So if
// t's fraction, RN(t - floor(t)) (exact, or within 2^-25 for t in (-1, 0)),
// lies in (B, 1 - B) with B = 2^-15, then x - u is more than
// B - 2^-25 - 6*2^-18 > 2^-25 away from every integer, and
// ceil(x - u) = ceil(t) = floor(t) + 1.  Anything else -- t within B of an
// integer, a NaN or an infinity -- is left to code_exact (about 1 value in
// 16000).
#pragma once

namespace ob {

constexpr float kCertain = 3.0517578125e-05f;     // B = 2^-15
constexpr float kCertainHi = 0.999969482421875f;  // 1 - 2^-15
constexpr float kNormalMin = 1.17549435e-38f;     // 2^-126

template <int QMAX>
__device__ __forceinline__ float code_exact(float g, float scale, float u) {
  constexpr float qmax = (float)QMAX;
  const float x = __fdiv_rn(g, scale);
  const float f = floorf(x);
  const float fr = __fsub_rn(x, f);
  float qf = __fadd_rn(f, (u < fr) ? 1.0f : 0.0f);
  qf = qf > qmax ? qmax : qf;
  qf = qf < -qmax ? -qmax : qf;
  if (qf != qf) qf = 0.0f;
  return qf;
}

// rcp: 1/scale correctly rounded, for a scale >= kNormalMin.  Returns the
// code; *certain is false where only code_exact may be used.
template <int QMAX>
__device__ __forceinline__ float code_fast(float g, float rcp, float u, bool* certain) {
  constexpr float qmax = (float)QMAX;
  const float t = __fsub_rn(__fmul_rn(g, rcp), u);
  const float ft = floorf(t);
  const float dt = __fsub_rn(t, ft);
  float q = __fadd_rn(ft, 1.0f);
  q = q > qmax ? qmax : q;
  q = q < -qmax ? -qmax : q;
  *certain = dt > kCertain && dt < kCertainHi;
  return q;
}

// 1/scale for code_fast, or 0 where every code must come from code_exact
// (scale 0, or below the normal range, or not finite).
__device__ __forceinline__ float code_rcp(float scale) {
  return scale >= kNormalMin ? __frcp_rn(scale) : 0.0f;
}

}  // namespace ob
