// Device arithmetic of the FP8 1x128 quantizer shared by the stand-alone
// quantizer kernel and the small-M kernel that quantizes its token rows
// itself, so that both produce the same codes and scale bytes bit for bit.
#pragma once

#include <cstdint>

#include "iq_internal.h"
#include "iq_ptx.cuh"

namespace iq {

// |x| of two packed BF16 values, as unsigned 16-bit lanes, max-reduced.
__device__ __forceinline__ uint32_t abs_max_bf16x2(uint32_t acc, uint32_t v) {
  return __vmaxu2(acc, v & 0x7FFF7FFFu);
}

// Scale exponent e of the FP8 stage: the smallest integer with
// 448 * 2^e >= max(amax, 1e-4).  With a = (1 + f) 2^E, 448 = 1.75 * 2^8:
// e = E - 8 when f <= 0.75 (mantissa bits <= 0x600000), else E - 7.
__device__ __forceinline__ int fp8_scale_exponent(float amax) {
  const float a = fmaxf(amax, kAmaxFloor);
  const uint32_t bits = __float_as_uint(a);
  const int E = static_cast<int>(bits >> 23) - 127;
  return E - 8 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
}

// 2^-e, exact.
__device__ __forceinline__ float fp8_inv_scale(int e) { return __uint_as_float(static_cast<uint32_t>(127 - e) << 23); }

// Two packed BF16 values -> two E4M3 codes of x * 2^-e (inv = 2^-e).
__device__ __forceinline__ uint32_t quant_pair(uint32_t bf2, float inv) {
  const float lo = __uint_as_float(bf2 << 16) * inv;
  const float hi = __uint_as_float(bf2 & 0xFFFF0000u) * inv;
  return cvt_e4m3x2(lo, hi);
}

__device__ __forceinline__ uint32_t quant_quad(uint32_t a, uint32_t b, float inv) {
  return quant_pair(a, inv) | (quant_pair(b, inv) << 16);
}

}  // namespace iq
