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

// NVFP4-style block scale: the E4M3 code of round-to-nearest(max(a, 1e-4) / 6)
// (an IEEE float32 division, then the hardware's E4M3 conversion), or code 1
// (2^-9, the smallest positive E4M3) when that rounds to zero; *s gets the
// scale's value.
__device__ __forceinline__ uint32_t nvfp4_scale_code(float a, float* s) {
  const float t = __fdiv_rn(fmaxf(a, kAmaxFloor), 6.0f);
  uint32_t code = cvt_e4m3x2(t, 0.f) & 0xFFu;
  if (code == 0u) code = 1u;
  *s = e4m3_to_float(code);
  return code;
}

// 2^-e / sqrt(128): multiplying an unscaled Hadamard output v by it gives
// fp32(z) * 2^-e with z = v / sqrt(128) (a power-of-two factor is exact).
__device__ __forceinline__ float fp4_code_factor(int e) {
  return __uint_as_float(static_cast<uint32_t>(127 - e) << 23) * kInvSqrt128;
}

}  // namespace iq
