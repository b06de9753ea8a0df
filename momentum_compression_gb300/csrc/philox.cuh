// Philox4x32-10, the counter-based generator of Salmon, Moraes, Dror and
// Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11): ten rounds of
// two 32x32->64-bit products with multipliers 0xD2511F53 and 0xCD9E8D57,
// the key advanced by 0x9E3779B9 and 0xBB67AE85 between rounds.  Used by the
// stochastic-rounding quantizers: the uniform of element k at call `step`
// is word k&3 of the output for counter (k>>2 low, k>>2 high, step low,
// step high), u = (word >> 8) * 2^-24.
#pragma once

#include <cstdint>

namespace ob {

// Round keys of Philox4x32-10: key k advanced by (0x9E3779B9, 0xBB67AE85)
// before every round but the first; computed once per thread, or once on
// the host and passed to a kernel as a parameter (its rounds then read the
// keys from the constant bank instead of holding 20 registers).
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};

__host__ __device__ __forceinline__ PhiloxKeys philox_keys(uint32_t k0, uint32_t k1) {
  PhiloxKeys K;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    K.k0[r] = k0 + (uint32_t)r * 0x9E3779B9u;
    K.k1[r] = k1 + (uint32_t)r * 0xBB67AE85u;
  }
  return K;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKeys& K) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ K.k0[r], (uint32_t)p1,
                   (uint32_t)(p0 >> 32) ^ c.w ^ K.k1[r], (uint32_t)p0);
  }
  return c;
}

// The same generator on two counters at once, round by round: two
// independent chains side by side in program order, so that one lane's
// dependent multiply-xor chains overlap.
__device__ __forceinline__ void philox4x32_10_x2(uint4& a, uint4& b, const PhiloxKeys& K) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t a0 = (uint64_t)0xD2511F53u * a.x;
    const uint64_t a1 = (uint64_t)0xCD9E8D57u * a.z;
    const uint64_t b0 = (uint64_t)0xD2511F53u * b.x;
    const uint64_t b1 = (uint64_t)0xCD9E8D57u * b.z;
    a = make_uint4((uint32_t)(a1 >> 32) ^ a.y ^ K.k0[r], (uint32_t)a1,
                   (uint32_t)(a0 >> 32) ^ a.w ^ K.k1[r], (uint32_t)a0);
    b = make_uint4((uint32_t)(b1 >> 32) ^ b.y ^ K.k0[r], (uint32_t)b1,
                   (uint32_t)(b0 >> 32) ^ b.w ^ K.k1[r], (uint32_t)b0);
  }
}

// Word c of a Philox output.
__device__ __forceinline__ uint32_t word_of(const uint4& u, int c) {
  return c == 0 ? u.x : c == 1 ? u.y : c == 2 ? u.z : u.w;
}

__device__ __forceinline__ float uniform_of(uint32_t word) {
  return __fmul_rn((float)(word >> 8), 5.9604644775390625e-08f);  // 2^-24
}

}  // namespace ob
