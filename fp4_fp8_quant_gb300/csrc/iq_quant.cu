// K1: the packed-UE8M0 FP8 1x128 online quantizer.
//
// Follows the TokenSpeed PR "perf(deepseek-v4): accelerate indexer Q and
// packed FP8 quantization" (Summary: packed-UE8M0 FP8 online quantizer for
// DeepGEMM activations; Risk and fallback: contiguous aligned BF16 input with
// K divisible by 128, the packed-UE8M0 scale contract, the tiny-scale floor)
// and the "FP8 input and UE8M0 scales" step of the TensorRT-LLM PR "Fuse
// DeepSeek-V4 Indexer Q projection with CuTe DSL" (sequence diagram).
//
// Design (HBM-bound, no reuse): one warp per (row, group of four 128-blocks).
// Each lane owns 16 consecutive BF16 values (two 16-byte loads), eight lanes
// form one 128-block, so a warp load instruction moves 512 contiguous bytes.
// The block amax is an integer max over the sign-cleared BF16 bit patterns
// (order-preserving for finite values) reduced with three shuffles; the scale
// exponent comes from the float32 exponent and mantissa bits of the floored
// amax; the E4M3 codes come from cvt.rn.satfinite on x * 2^-e, which is exact
// before rounding.  Lane 0 gathers the four scale bytes into one int32 word of
// the M-major packed layout.  Rows past M (up to the multiple of 4) get zero
// words, so the kernel writes the whole scale array.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "iq_fp8.cuh"
#include "iq_internal.h"
#include "iq_ptx.cuh"

namespace iq {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__global__ void __launch_bounds__(kThreads) quant_1x128_kernel(const uint16_t* __restrict__ x, int M, int K,
                                                               long long ldx, uint8_t* __restrict__ y,
                                                               long long ldy, int32_t* __restrict__ sf, int m_al,
                                                               int groups) {
  // The fused GEMM that usually follows may be scheduled now; it waits for
  // this grid's completion before reading anything.
  grid_launch_dependents();
  const long long unit = (static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (unit >= static_cast<long long>(m_al) * groups) return;
  const int row = static_cast<int>(unit / groups);
  const int g = static_cast<int>(unit - static_cast<long long>(row) * groups);
  const int col = g * 512 + lane * 16;
  const bool active = row < M && col < K;

  uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
  const uint16_t* src = x + row * ldx + col;
  if (active) {
    a = ld_stream(src);
    b = ld_stream(src + 8);
  }
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
  if (active) {
    uint4 out;
    out.x = quant_quad(a.x, a.y, inv);
    out.y = quant_quad(a.z, a.w, inv);
    out.z = quant_quad(b.x, b.y, inv);
    out.w = quant_quad(b.z, b.w, inv);
    *reinterpret_cast<uint4*>(y + row * ldy + col) = out;
  }
  const uint32_t byte = active ? static_cast<uint32_t>(e + 127) : 0u;
  const uint32_t b0 = __shfl_sync(0xFFFFFFFFu, byte, 0);
  const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, byte, 8);
  const uint32_t b2 = __shfl_sync(0xFFFFFFFFu, byte, 16);
  const uint32_t b3 = __shfl_sync(0xFFFFFFFFu, byte, 24);
  if (lane == 0) sf[static_cast<long long>(g) * m_al + row] = static_cast<int32_t>(b0 | (b1 << 8) | (b2 << 16) | (b3 << 24));
}

}  // namespace

cudaError_t launch_quant_1x128(const void* x, int M, int K, long long ldx, void* y, long long ldy, int32_t* sf,
                               cudaStream_t stream) {
  const int m_al = (M + 3) / 4 * 4;
  const int groups = (K + 511) / 512;
  const long long warps = static_cast<long long>(m_al) * groups;
  const long long blocks = (warps * 32 + kThreads - 1) / kThreads;
  quant_1x128_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
      static_cast<const uint16_t*>(x), M, K, ldx, static_cast<uint8_t*>(y), ldy, sf, m_al, groups);
  return cudaGetLastError();
}

}  // namespace iq
