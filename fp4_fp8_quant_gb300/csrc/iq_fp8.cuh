// Device arithmetic of the FP8 1x128 quantizer, shared by the stand-alone
// quantizer kernel and the CTA-pair GEMM kernel that quantizes its token rows
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

// Streaming 16-byte load of data no kernel writes while this one runs (the
// BF16 token rows): read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// One unit of the quantizer, by a whole warp: 512 consecutive columns (four
// 128-blocks) of one row.  Lane l holds columns 16l..16l+15 as two 16-byte
// words a, b (zero when !active), so eight lanes form one 128-block.  The
// block amax is an integer max over the sign-cleared BF16 patterns (order
// preserving for finite values), reduced over the eight lanes; the E4M3 codes
// of x * 2^-e go to `codes`; the return value, the same in every lane, is the
// unit's packed scale word (byte j = e + 127 of block j, 0 for inactive
// blocks).  All 32 lanes must take part.
__device__ __forceinline__ uint32_t fp8_quant_unit(const uint4& a, const uint4& b, bool active, uint4& codes) {
  uint32_t m2 = abs_max_bf16x2(0u, a.x);
  m2 = abs_max_bf16x2(m2, a.y);
  m2 = abs_max_bf16x2(m2, a.z);
  m2 = abs_max_bf16x2(m2, a.w);
  m2 = abs_max_bf16x2(m2, b.x);
  m2 = abs_max_bf16x2(m2, b.y);
  m2 = abs_max_bf16x2(m2, b.z);
  m2 = abs_max_bf16x2(m2, b.w);
  uint32_t m1 = max(m2 & 0xFFFFu, m2 >> 16);
  m1 = max(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, 1));
  m1 = max(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, 2));
  m1 = max(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, 4));
  const float amax = __uint_as_float(m1 << 16);
  const int e = fp8_scale_exponent(amax);
  const float inv = fp8_inv_scale(e);
  codes.x = quant_quad(a.x, a.y, inv);
  codes.y = quant_quad(a.z, a.w, inv);
  codes.z = quant_quad(b.x, b.y, inv);
  codes.w = quant_quad(b.z, b.w, inv);
  const uint32_t byte = active ? static_cast<uint32_t>(e + 127) : 0u;
  const uint32_t b0 = __shfl_sync(0xFFFFFFFFu, byte, 0);
  const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, byte, 8);
  const uint32_t b2 = __shfl_sync(0xFFFFFFFFu, byte, 16);
  const uint32_t b3 = __shfl_sync(0xFFFFFFFFu, byte, 24);
  return b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
}

}  // namespace iq
