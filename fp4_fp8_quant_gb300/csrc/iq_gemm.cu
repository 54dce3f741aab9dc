// K2: block-scaled FP8 GEMM with the indexer-Q epilogue fused in
// (RoPE -> Hadamard-128 -> FP4 E2M1 with 1x32 UE8M0 scales).
//
// What it computes follows the TensorRT-LLM PR "Fuse DeepSeek-V4 Indexer Q
// projection with CuTe DSL" (sequence diagram: the GEMM runs on the FP8 input
// and UE8M0 scales and its epilogue does RoPE and FP4, returning packed FP4 Q
// and scales; review comment on the fused epilogue: MXF8 with scale vector 32
// and a 128-column MMA tile per head, and every scale must be applied) and the
// TokenSpeed PR "perf(deepseek-v4): accelerate indexer Q and packed FP8
// quantization" (Summary: RoPE, Hadamard and fusedCat FP4 on the indexer Q).
//
// Tile: 128 tokens x 256 output features (two heads) per CTA tile, K = 1536 in
// twelve 128-byte K-blocks.  Persistent CTAs (one per SM) walk the tiles.
// Warp roles (320 threads):
//   warp 0      TMA producer: a 4-stage ring of {X tile 16 KB, W tile 32 KB},
//               128-byte swizzled, plus the per-tile scale factors staged in
//               shared memory in the layout tcgen05.cp 32x128b expects;
//   warp 1      TMEM owner and MMA issuer: copies the scale factors into TMEM
//               and issues tcgen05.mma kind::mxf8f6f4 block_scale (scale vector
//               1X = one UE8M0 per 32 K) into a 128 x 256 FP32 accumulator;
//   warps 2..9  epilogue: each thread owns one (token, head) pair = one TMEM
//               lane x 128 columns.  It drains its 128 values to registers,
//               releases the accumulator at once so the next tile's MMAs can
//               start, then does RoPE, the in-register 128-point fast
//               Walsh-Hadamard transform, the FP4 block quantization and the
//               stores.  The FP32 pre-quant Q never touches memory unless the
//               debug output is requested.
//
// Scale factors.  The activation scales are per 1x128 block and the weight
// scales per 128x128 block, but the MMA applies one scale per 32 K: every
// 32-wide K step of a 128-block uses the same byte, selected by the scale-ID
// field of the instruction descriptor (kb % 4 picks the byte of the packed
// word that holds 4 consecutive K-blocks).  This is exact: the scales are
// powers of two.
//
// Every mbarrier wait is bounded (GemmArgs::timeout_ns); a wait that gives up
// records its kind in the device status word, raises a CTA-wide abort flag so
// the other roles leave their loops, and the teardown waits (bounded) for the
// CTA's own TMA loads and tcgen05 operations before TMEM is freed.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "iq_internal.h"
#include "iq_ptx.cuh"

namespace iq {

__device__ uint32_t g_iq_status;

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK;                 // 16 KB
constexpr int kBBytes = BN * BK;                 // 32 KB
constexpr int kStageTx = kABytes + kBBytes;
constexpr int kNumEpiWarps = 8;
constexpr int kThreads = (2 + kNumEpiWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;
constexpr uint32_t kSfaCol = 256;                // + 8 g, 4 columns each
constexpr uint32_t kSfbCol = 288;                // + 8 g, 8 columns each (two 128-row halves)

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kSfaWords = kScaleGroups * 128;    // per buffer
constexpr int kSfbWords = kScaleGroups * 256;
constexpr int kOffSfa = kOffB + kStages * kBBytes;
constexpr int kOffSfb = kOffSfa + 2 * kSfaWords * 4;
constexpr int kOffBar = kOffSfb + 2 * kSfbWords * 4;
constexpr int kNumBars = 2 * kStages + 4 + 3;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack

constexpr float kInvSqrt128 = 0.0883883476483184405501f;
constexpr float kTwoPi = 6.28318530717958647692f;

__device__ __forceinline__ void fail(volatile uint32_t* abort_flag, uint32_t bit) {
  atomicOr(&g_iq_status, bit);
  *abort_flag = 1u;
}

// Scale exponent of the FP4 stage: smallest e with 6 * 2^e >= max(a, 1e-4).
// With a = (1 + f) 2^E and 6 = 1.5 * 2^2: e = E - 2 when f <= 0.5, else E - 1.
__device__ __forceinline__ int fp4_scale_exponent(float a) {
  a = fmaxf(a, kAmaxFloor);
  const uint32_t bits = __float_as_uint(a);
  const int E = static_cast<int>(bits >> 23) - 127;
  return E - 2 + ((bits & 0x7FFFFFu) > 0x400000u ? 1 : 0);
}

// RoPE, Hadamard, FP4 for one (token, head): v holds the 128 FP32 GEMM outputs.
__device__ __forceinline__ void epilogue_row(float (&v)[128], int row, int head, const GemmArgs& args) {
  // NeoX RoPE on dims 0..63: pairs (i, i+32), angle = pos * 10000^(-i/32).
  // The angle is reduced in turns with a two-float product so that it stays
  // accurate for large positions; the reduced angle lies in [-pi, pi].
  const float p = static_cast<float>(args.pos[row]);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float th = p * args.rope.hi[i];
    float tl = fmaf(p, args.rope.hi[i], -th);
    tl = fmaf(p, args.rope.lo[i], tl);
    const float fr = (th - rintf(th)) + tl;
    float s, c;
    __sincosf(fr * kTwoPi, &s, &c);
    const float x1 = v[i], x2 = v[i + 32];
    v[i] = x1 * c - x2 * s;
    v[i + 32] = x2 * c + x1 * s;
  }
  // Fast Walsh-Hadamard transform in Sylvester order (unscaled).
#pragma unroll
  for (int h = 1; h < 128; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 128; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
    }
  }
  // FP4: z = v / sqrt(128); per 32-block scale e; codes = E2M1(z * 2^-e).
  // z * 2^-e is formed as v * (2^-e / sqrt(128)), equal to fp32(z) * 2^-e.
  uint32_t codes[16];
  uint32_t sfw = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[32 * b + j]));
    const int e = fp4_scale_exponent(amax * kInvSqrt128);
    const float k = __uint_as_float(static_cast<uint32_t>(127 - e) << 23) * kInvSqrt128;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      float q[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) q[j] = v[32 * b + 8 * t + j] * k;
      codes[4 * b + t] = cvt_e2m1x8(q);
    }
    sfw |= static_cast<uint32_t>(e + 127) << (8 * b);
  }
  uint4* dst = reinterpret_cast<uint4*>(args.q_fp4 + static_cast<long long>(row) * (kQDim / 2) + head * 64);
#pragma unroll
  for (int t = 0; t < 4; ++t)
    dst[t] = make_uint4(codes[4 * t], codes[4 * t + 1], codes[4 * t + 2], codes[4 * t + 3]);
  *reinterpret_cast<uint32_t*>(args.q_sf + static_cast<long long>(row) * (kQDim / 32) + head * 4) = sfw;
  if (args.q_pre != nullptr) {
    float4* pre = reinterpret_cast<float4*>(args.q_pre + static_cast<long long>(row) * kQDim + head * kHeadDim);
#pragma unroll
    for (int t = 0; t < 32; ++t)
      pre[t] = make_float4(v[4 * t] * kInvSqrt128, v[4 * t + 1] * kInvSqrt128, v[4 * t + 2] * kInvSqrt128,
                           v[4 * t + 3] * kInvSqrt128);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_rope_hadamard_fp4_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                                  const __grid_constant__ GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem + kOffA;
  uint8_t* sB = smem + kOffB;
  uint32_t* sSfa = reinterpret_cast<uint32_t*>(smem + kOffSfa);
  uint32_t* sSfb = reinterpret_cast<uint32_t*>(smem + kOffSfb);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* sf_full = bars + 2 * kStages;
  uint64_t* sf_empty = sf_full + 2;
  uint64_t* tmem_full = sf_empty + 2;
  uint64_t* tmem_empty = tmem_full + 1;
  uint64_t* final_bar = tmem_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t timeout = args.timeout_ns;

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sf_full[b], 1);
      mbar_init(&sf_empty[b], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, kNumEpiWarps);
    mbar_init(final_bar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const int num_m_tiles = args.num_m_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0;
    uint32_t issued_mask = 0, issued_phase = 0;   // per stage: a load was issued / its phase
    int local = 0;
    for (int tile = blockIdx.x; tile < args.num_tiles; tile += gridDim.x, ++local) {
      // Every exit decision is made warp-uniform: the lanes must stay
      // converged for the shuffles below.
      if (__any_sync(0xFFFFFFFFu, *abort_flag != 0u)) break;
      const int m0 = (tile % num_m_tiles) * BM;
      const int n_tile = tile / num_m_tiles;
      const int buf = local & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sf_empty[buf], ((local >> 1) & 1) ^ 1, timeout))) {
        if (lane == 0) fail(abort_flag, kStatusProducerWait);
        break;
      }
      // Scale factors in the tcgen05.cp 32x128b layout: word [r * 4 + c] of a
      // 128-row tile holds row c * 32 + r.
      uint32_t* sfa = sSfa + buf * kSfaWords;
      uint32_t* sfb = sSfb + buf * kSfbWords;
#pragma unroll
      for (int g = 0; g < kScaleGroups; ++g) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int m = m0 + c * 32 + lane;
          sfa[g * 128 + lane * 4 + c] =
              m < args.m_al ? static_cast<uint32_t>(__ldg(args.x_sf + static_cast<long long>(g) * args.m_al + m)) : 0u;
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint8_t* ws = args.w_sf + (n_tile * 2 + half) * kNumKBlocks + 4 * g;
          const uint32_t word = static_cast<uint32_t>(__ldg(ws)) | (static_cast<uint32_t>(__ldg(ws + 1)) << 8) |
                                (static_cast<uint32_t>(__ldg(ws + 2)) << 16) |
                                (static_cast<uint32_t>(__ldg(ws + 3)) << 24);
#pragma unroll
          for (int c = 0; c < 4; ++c) sfb[g * 256 + half * 128 + lane * 4 + c] = word;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      bool ok = true;
      if (lane == 0) {
        mbar_arrive(&sf_full[buf]);
        for (int kb = 0; kb < kNumKBlocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, timeout)) {
            fail(abort_flag, kStatusProducerWait);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], kStageTx);
          tma_load_2d(sA + stage * kABytes, &tm_x, &full[stage], kb * BK, m0);
          tma_load_2d(sB + stage * kBBytes, &tm_w, &full[stage], kb * BK, n_tile * BN);
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
    }
    // Teardown: the last load issued into each stage must have landed before
    // the shared memory can be released.
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        if ((issued_mask >> s) & 1u) {
          if (!mbar_wait(&full[s], (issued_phase >> s) & 1u, timeout)) fail(abort_flag, kStatusTeardownWait);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < args.num_tiles && ok; tile += gridDim.x, ++local) {
        if (*abort_flag) break;
        const int buf = local & 1;
        if (!mbar_wait(&sf_full[buf], (local >> 1) & 1, timeout) ||
            !mbar_wait(tmem_empty, (local & 1) ^ 1, timeout)) {
          fail(abort_flag, kStatusMmaWait);
          break;
        }
        tc_fence_after_sync();
        const uint32_t* sfa = sSfa + buf * kSfaWords;
        const uint32_t* sfb = sSfb + buf * kSfbWords;
#pragma unroll
        for (int g = 0; g < kScaleGroups; ++g) {
          tc_cp_32x128b_warpx4(tmem + kSfaCol + 8 * g, smem_desc_sf(smem_u32(sfa + g * 128)));
          tc_cp_32x128b_warpx4(tmem + kSfbCol + 8 * g, smem_desc_sf(smem_u32(sfb + g * 256)));
          tc_cp_32x128b_warpx4(tmem + kSfbCol + 8 * g + 4, smem_desc_sf(smem_u32(sfb + g * 256 + 128)));
        }
        tc_commit(&sf_empty[buf]);
        for (int kb = 0; kb < kNumKBlocks; ++kb) {
          if (*abort_flag || !mbar_wait(&full[stage], phase, timeout)) {
            fail(abort_flag, kStatusMmaWait);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t adesc = smem_desc_sw128(smem_u32(sA + stage * kABytes));
          const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + stage * kBBytes));
          const uint32_t idesc = idesc_mxf8_e4m3(BM, BN, kb & 3, kb & 3);
          const uint32_t sfa_t = tmem + kSfaCol + 8 * (kb >> 2);
          const uint32_t sfb_t = tmem + kSfbCol + 8 * (kb >> 2);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k) {
            // advance 32 bytes along K inside the 128-byte swizzle atom
            tc_mma_mxf8(tmem + kAccCol, adesc + 2 * k, bdesc + 2 * k, idesc, sfa_t, sfb_t, (kb | k) != 0);
          }
          tc_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) tc_commit(tmem_full);
      }
      // Teardown: every tcgen05 operation of this thread has completed.
      tc_commit(final_bar);
      if (!mbar_wait(final_bar, 0, timeout)) fail(abort_flag, kStatusTeardownWait);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;            // the TMEM lane group this warp may read
    const int half = (warp - 2) >> 2;     // which head of the tile
    int local = 0;
    for (int tile = blockIdx.x; tile < args.num_tiles; tile += gridDim.x, ++local) {
      // Warp-uniform exit decisions: tcgen05.ld below is .sync.aligned.
      if (__any_sync(0xFFFFFFFFu, *abort_flag != 0u)) break;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(tmem_full, local & 1, timeout))) {
        if (lane == 0) fail(abort_flag, kStatusEpilogueWait);
        break;
      }
      tc_fence_after_sync();
      float v[128];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + kAccCol + half * 128;
      tmem_ld_32x32b_x32(taddr + 0, v + 0);
      tmem_ld_32x32b_x32(taddr + 32, v + 32);
      tmem_ld_32x32b_x32(taddr + 64, v + 64);
      tmem_ld_32x32b_x32(taddr + 96, v + 96);
      tmem_ld_wait(v + 0);
      tmem_ld_wait(v + 32);
      tmem_ld_wait(v + 64);
      tmem_ld_wait(v + 96);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_empty);
      const int row = (tile % num_m_tiles) * BM + quad * 32 + lane;
      const int head = (tile / num_m_tiles) * 2 + half;
      if (row < args.M) epilogue_row(v, row, head, args);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int gemm_smem_bytes() { return kSmemBytes; }

cudaError_t gemm_setup_device() {
  return cudaFuncSetAttribute(gemm_rope_hadamard_fp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemBytes);
}

cudaError_t launch_gemm_rope_hadamard_fp4(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const GemmArgs& args,
                                          int num_sms, cudaStream_t stream) {
  const int grid = args.num_tiles < num_sms ? args.num_tiles : num_sms;
  gemm_rope_hadamard_fp4_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tm_x, tm_w, args);
  return cudaGetLastError();
}

cudaError_t read_device_status(uint32_t* flags, bool reset) {
  uint32_t v = 0;
  cudaError_t err = cudaMemcpyFromSymbol(&v, g_iq_status, sizeof(v));
  if (err != cudaSuccess) return err;
  if (flags) *flags = v;
  if (reset) {
    const uint32_t zero = 0;
    err = cudaMemcpyToSymbol(g_iq_status, &zero, sizeof(zero));
  }
  return err;
}

}  // namespace iq
