// Device arithmetic of the FP4 stage shared by the fused GEMM kernels (the
// large-M CTA-pair kernel and the small-M swapped-operand kernel), so that
// both routes take the FP4 scale decision by the same rule.
#pragma once

#include <cstdint>

#include "iq_internal.h"

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

// 2^-e / sqrt(128): multiplying an unscaled Hadamard output v by it gives
// fp32(z) * 2^-e with z = v / sqrt(128) (a power-of-two factor is exact).
__device__ __forceinline__ float fp4_code_factor(int e) {
  return __uint_as_float(static_cast<uint32_t>(127 - e) << 23) * kInvSqrt128;
}

}  // namespace iq
