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
//
// Host-rows variant (the host-buffer entry's quantizer, reading its rows from
// page-locked host memory): there a half-used sector costs a whole transfer
// over the host link, and the map above, whose two loads per lane each use
// half of every sector they touch, reads at half the link's rate.  The
// variant gives lane l columns 8l..8l+7 and 256+8l..256+8l+7 of the unit, so
// each warp load reads 512 contiguous bytes (16 lanes per block, the two
// blocks of a lane reduced together in one packed word), loops over units
// with a grid of one block per SM (it runs beside the GEMM kernel), and also
// copies the rows' positions.  From HBM the first map is the faster one.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "iq_fp8.cuh"
#include "iq_internal.h"
#include "iq_ptx.cuh"

namespace iq {

namespace {

constexpr int kThreads = 256;
// Host-rows variant: 128 threads (4K registers) per block, so that two of its
// blocks fit on an SM beside a CTA of the GEMM kernel (53.8K registers, 224 KB
// of shared memory; each further block reserves 1 KB) whatever way the
// blocks are spread; one block per SM keeps ~0.6 MB of loads in flight.
constexpr int kHostThreads = 128;

__global__ void __launch_bounds__(kThreads) quant_1x128_kernel(const uint16_t* __restrict__ x, int M, int K,
                                                               long long ldx, uint8_t* __restrict__ y,
                                                               long long ldy, int32_t* __restrict__ sf, int m_al,
                                                               int groups) {
  // The fused GEMM that usually follows may be scheduled now; it waits for
  // this grid's completion before reading anything.  This kernel is itself
  // launched as a programmatic dependent of whatever precedes it in the
  // stream, so its blocks may be resident before that kernel ends: nothing
  // is read or written before the dependency wait.
  grid_launch_dependents();
  grid_dependency_wait();
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
    a = ld_stream_v4(src);
    b = ld_stream_v4(src + 8);
  }
  uint4 out;
  const uint32_t word = fp8_quant_unit(a, b, active, out);
  if (active) *reinterpret_cast<uint4*>(y + row * ldy + col) = out;
  if (lane == 0) sf[static_cast<long long>(g) * m_al + row] = static_cast<int32_t>(word);
}

__global__ void __launch_bounds__(kHostThreads)
    quant_1x128_host_rows_kernel(const uint16_t* __restrict__ x, int M, int K, long long ldx, uint8_t* __restrict__ y,
                                 long long ldy, int32_t* __restrict__ sf, int m_al, int groups,
                                 const int32_t* __restrict__ pos_src, int32_t* __restrict__ pos_dst) {
  const int lane = threadIdx.x & 31;
  const long long units = static_cast<long long>(m_al) * groups;
  const long long stride = static_cast<long long>(gridDim.x) * (kHostThreads / 32);
  // A grid smaller than the unit count loops, which bounds how many threads
  // and registers the kernel holds on each SM beside the GEMM kernel.
  for (long long unit = (static_cast<long long>(blockIdx.x) * kHostThreads + threadIdx.x) >> 5; unit < units;
       unit += stride) {
    const int row = static_cast<int>(unit / groups);
    const int g = static_cast<int>(unit - static_cast<long long>(row) * groups);
    // Lane l holds elements 8l..8l+7 (block l/16) and 256+8l..256+8l+7
    // (block 2 + l/16) of the unit's 512 columns, so each warp load reads
    // 512 contiguous bytes: whole sectors, also from host memory.
    const int half = lane >> 4;
    const int col_a = g * 512 + lane * 8, col_b = col_a + 256;
    const bool active_a = row < M && g * 512 + half * 128 < K;
    const bool active_b = row < M && g * 512 + 256 + half * 128 < K;
    // The rows' positions are copied too; the store waits for the load only
    // at the end of the unit.
    const bool copy_pos = g == 0 && lane == 0 && row < M;
    const int32_t pos = copy_pos ? pos_src[row] : 0;

    uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
    const uint16_t* src = x + row * ldx;
    if (active_a) a = ld_stream_v4(src + col_a);
    if (active_b) b = ld_stream_v4(src + col_b);
    uint32_t ma = abs_max_bf16x2(0u, a.x);
    ma = abs_max_bf16x2(ma, a.y);
    ma = abs_max_bf16x2(ma, a.z);
    ma = abs_max_bf16x2(ma, a.w);
    uint32_t mb = abs_max_bf16x2(0u, b.x);
    mb = abs_max_bf16x2(mb, b.y);
    mb = abs_max_bf16x2(mb, b.z);
    mb = abs_max_bf16x2(mb, b.w);
    // Low half: this lane's block-a maximum; high half: its block-b maximum;
    // reduced over the 16 lanes of each block.
    uint32_t m2 = max(ma & 0xFFFFu, ma >> 16) | (max(mb & 0xFFFFu, mb >> 16) << 16);
    m2 = __vmaxu2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, 1));
    m2 = __vmaxu2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, 2));
    m2 = __vmaxu2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, 4));
    m2 = __vmaxu2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, 8));

    const int e_a = fp8_scale_exponent(__uint_as_float(m2 << 16));
    const int e_b = fp8_scale_exponent(__uint_as_float(m2 & 0xFFFF0000u));
    uint8_t* dst = y + row * ldy;
    if (active_a) {
      const float inv = fp8_inv_scale(e_a);
      *reinterpret_cast<uint2*>(dst + col_a) = make_uint2(quant_quad(a.x, a.y, inv), quant_quad(a.z, a.w, inv));
    }
    if (active_b) {
      const float inv = fp8_inv_scale(e_b);
      *reinterpret_cast<uint2*>(dst + col_b) = make_uint2(quant_quad(b.x, b.y, inv), quant_quad(b.z, b.w, inv));
    }
    // Scale bytes of blocks 0..3: e_a of lanes 0 and 16, e_b of lanes 0 and 16.
    const uint32_t byte_a = active_a ? static_cast<uint32_t>(e_a + 127) : 0u;
    const uint32_t byte_b = active_b ? static_cast<uint32_t>(e_b + 127) : 0u;
    const uint32_t pair = byte_a | (byte_b << 16);
    const uint32_t pair16 = __shfl_sync(0xFFFFFFFFu, pair, 16);
    const uint32_t b0 = pair & 0xFFu, b2 = pair >> 16;
    const uint32_t b1 = pair16 & 0xFFu, b3 = pair16 >> 16;
    if (lane == 0) {
      sf[static_cast<long long>(g) * m_al + row] = static_cast<int32_t>(b0 | (b1 << 8) | (b2 << 16) | (b3 << 24));
    }
    if (copy_pos) pos_dst[row] = pos;
  }
}


// The FP4 stage's element conversion alone (the one both fused GEMM kernels
// use): eight floats per thread through cvt_e2m1x8, one code per output byte.
__global__ void e2m1_codes_kernel(const float* __restrict__ x, long long n8, uint8_t* __restrict__ out) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(x)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(x)[2 * i + 1];
  const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  const uint32_t c = cvt_e2m1x8(v);
  uint2 o;
  o.x = (c & 0xFu) | ((c >> 4) & 0xFu) << 8 | ((c >> 8) & 0xFu) << 16 | ((c >> 12) & 0xFu) << 24;
  o.y = ((c >> 16) & 0xFu) | ((c >> 20) & 0xFu) << 8 | ((c >> 24) & 0xFu) << 16 | ((c >> 28) & 0xFu) << 24;
  reinterpret_cast<uint2*>(out)[i] = o;
}

}  // namespace

cudaError_t launch_e2m1_codes(const float* x, long long n, uint8_t* codes, cudaStream_t stream) {
  const long long n8 = n / 8;
  const long long blocks = (n8 + 255) / 256;
  e2m1_codes_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, n8, codes);
  return cudaGetLastError();
}

cudaError_t launch_quant_1x128(const void* x, int M, int K, long long ldx, void* y, long long ldy, int32_t* sf,
                               cudaStream_t stream) {
  const int m_al = (M + 3) / 4 * 4;
  const int groups = (K + 511) / 512;
  const long long warps = static_cast<long long>(m_al) * groups;
  const long long blocks = (warps * 32 + kThreads - 1) / kThreads;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quant_1x128_kernel, static_cast<const uint16_t*>(x), M, K, ldx,
                            static_cast<uint8_t*>(y), ldy, sf, m_al, groups);
}

cudaError_t launch_quant_1x128_host_rows(const void* x, int M, int K, long long ldx, void* y, long long ldy,
                                         int32_t* sf, const int32_t* pos_src, int32_t* pos_dst, int max_blocks,
                                         cudaStream_t stream) {
  const int m_al = (M + 3) / 4 * 4;
  const int groups = (K + 511) / 512;
  const long long warps = static_cast<long long>(m_al) * groups;
  long long blocks = (warps * 32 + kHostThreads - 1) / kHostThreads;
  if (max_blocks > 0 && blocks > max_blocks) blocks = max_blocks;
  quant_1x128_host_rows_kernel<<<static_cast<unsigned>(blocks), kHostThreads, 0, stream>>>(
      static_cast<const uint16_t*>(x), M, K, ldx, static_cast<uint8_t*>(y), ldy, sf, m_al, groups, pos_src, pos_dst);
  return cudaGetLastError();
}

}  // namespace iq
