// Device arithmetic of the FP4 stage shared by the fused GEMM kernels (the
// large-M CTA-pair kernel and the small-M swapped-operand kernel), so that
// both routes take the FP4 scale decision by the same rule.
#pragma once

#include <cstdint>

#include "iq_internal.h"
#include "iq_ptx.cuh"

namespace iq {

constexpr float kInvSqrt128 = 0.0883883476483184405501f;
constexpr float kTwoPi = 6.28318530717958647692f;

// Scale exponent of the FP4 stage: smallest e with 6 * 2^e >= max(a, 1e-4).
// With a = (1 + f) 2^E and 6 = 1.5 * 2^2: e = E - 2 when f <= 0.5, else E - 1.
__device__ __forceinline__ int fp4_scale_exponent(float a) {
  a = fmaxf(a, kAmaxFloor);
  const uint32_t bits = __float_as_uint(a);
  const int E = static_cast<int>(bits >> 23) - 127;
  return E - 2 + ((bits & 0x7FFFFFu) > 0x400000u ? 1 : 0);
}

// OCP MX shared exponent of an E2M1 block: floor(log2(max(a, 1e-4))) - 2
// (emax of E2M1 is 2): the exponent field of the float minus 2.
__device__ __forceinline__ int fp4_scale_exponent_ocp(float a) {
  a = fmaxf(a, kAmaxFloor);
  return static_cast<int>(__float_as_uint(a) >> 23) - 127 - 2;
}

template <int kFmt>
__device__ __forceinline__ int fp4_block_exponent(float a) {
  if constexpr (kFmt == kFp4MxOcp) {
    return fp4_scale_exponent_ocp(a);
  } else {
    return fp4_scale_exponent(a);
  }
}

// float32(1/6): the NVFP4-style block scale target is amax / 6, formed as a
// product (it can differ from the correctly rounded quotient by one ulp, which
// moves the E4M3 decision only next to an E4M3 rounding midpoint).
constexpr float kSixth = 0x1.555556p-3f;

// E4M3 code of round-to-nearest(t) for a block scale target t >= 0, or code 1
// (2^-9, the smallest positive E4M3) when t rounds to zero.
__device__ __forceinline__ uint32_t nvfp4_code(float t) {
  const uint32_t code = cvt_e4m3x2(t, 0.f) & 0xFFu;
  return code == 0u ? 1u : code;
}

// Correctly rounded float32 reciprocal of a positive E4M3 value, from its
// code: 1 / ((1 + m/8) 2^(E-7)) = float32(8 / (8 + m)) * 2^(7-E) for normal
// codes, 1 / (m 2^-9) = float32(1 / m) * 2^9 for subnormal ones; each constant
// is the correctly rounded reciprocal and the power-of-two factor is applied
// exactly to its exponent field.
__device__ __forceinline__ uint32_t select8(uint32_t m, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3,
                                            uint32_t v4, uint32_t v5, uint32_t v6, uint32_t v7) {
  // Register-only choice among eight constants (an indexed array would be
  // placed in local memory).
  const uint32_t a = (m & 1u) ? v1 : v0, b = (m & 1u) ? v3 : v2;
  const uint32_t c = (m & 1u) ? v5 : v4, d = (m & 1u) ? v7 : v6;
  const uint32_t lo = (m & 2u) ? b : a, hi = (m & 2u) ? d : c;
  return (m & 4u) ? hi : lo;
}

__device__ __forceinline__ float e4m3_reciprocal(uint32_t code) {
  const uint32_t m = code & 7u;
  const int E = static_cast<int>((code >> 3) & 15u);
  if (E == 0)
    return __uint_as_float(select8(m, 0u, 0x3F800000u, 0x3F000000u, 0x3EAAAAABu, 0x3E800000u, 0x3E4CCCCDu,
                                   0x3E2AAAABu, 0x3E124925u) +
                           (9u << 23));
  const uint32_t inv_mant = select8(m, 0x3F800000u, 0x3F638E39u, 0x3F4CCCCDu, 0x3F3A2E8Cu, 0x3F2AAAABu, 0x3F1D89D9u,
                                    0x3F124925u, 0x3F088889u);
  return __uint_as_float(static_cast<uint32_t>(static_cast<int>(inv_mant) + ((7 - E) << 23)));
}

// 2^-e / sqrt(128): multiplying an unscaled Hadamard output v by it gives
// fp32(z) * 2^-e with z = v / sqrt(128) (a power-of-two factor is exact).
__device__ __forceinline__ float fp4_code_factor(int e) {
  return __uint_as_float(static_cast<uint32_t>(127 - e) << 23) * kInvSqrt128;
}

}  // namespace iq
