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
// CTA pairs.  The kernel runs in clusters of two CTAs (one per SM) that
// compute one 256-token x 256-feature (two heads) tile together with the
// 2-SM form of the MMA (tcgen05 cta_group::2, M = 256): each CTA holds its own
// 128 token rows of X and the 128 rows of W of one of the two heads, and its
// tensor memory receives the 128 x 256 FP32 accumulator of its own rows.  On
// GB300 the 1-SM M = 128 MMA measured 1.3-1.6x slower per SM than this form,
// which reaches the tensor-core peak.  K = 1536 streams as twelve 128-byte
// K-blocks.  Each pair takes a contiguous run of tiles, by default in
// token-major order (consecutive tiles share their token rows).  Up to 256
// tokens the tile is one head wide (128 features, each CTA loading 64 W rows
// of the head), so that twice as many pairs share the work.
// Warp roles (320 threads per CTA):
//   warp 0      TMA producer (both CTAs): a 6-stage ring of {X 16 KB, W 16 KB},
//               128-byte swizzled; each load signals the leader CTA's barrier.
//               It also stages the tile's scale factors in shared memory in
//               the layout tcgen05.cp 32x128b expects;
//   warp 1      TMEM owner (both CTAs) and, in the leader CTA, MMA issuer: it
//               copies the scale factors into both CTAs' tensor memories and
//               issues tcgen05.mma kind::mxf8f6f4 block_scale (scale vector 1X =
//               one UE8M0 per 32 K) for the pair;
//   warps 2..9  epilogue: each thread owns one (token, head) pair = one TMEM
//               lane x 128 columns.  It drains its 128 values to registers,
//               releases the accumulator at once, then does RoPE, the 128-point
//               fast Walsh-Hadamard transform and the FP4 block quantization in
//               packed FP32x2 arithmetic (scalar FP32 add/mul/fma next to the
//               MMAs slow the tensor pipe on GB300; the packed forms do not),
//               and stages the FP4 codes in shared memory, from where two bulk
//               tensor stores per tile write them.  The FP32 pre-quant Q never
//               touches memory unless the debug output is requested.  With
//               one-head tiles two warps share each (token, head): each
//               transforms one half of the dims in place in tensor memory and
//               reads the other half back for the last Hadamard stage.
//
// Scale factors.  The activation scales are per 1x128 block and the weight
// scales per 128x128 block, but the MMA applies one scale per 32 K: every
// 32-wide K step of a 128-block uses the same byte, selected by the scale-ID
// field of the instruction descriptor (kb % 4 picks the byte of the packed
// word that holds 4 consecutive K-blocks).  This is exact: the scales are
// powers of two.
//
// Every mbarrier wait is bounded (GemmArgs::timeout_ns); a wait that gives up
// records its kind in the device status word and raises a CTA abort flag so
// the other roles leave their loops; the epilogue warps take their exit
// decision together.  The teardown waits (bounded) until the pair's MMAs have
// released every stage this CTA loaded and completed, and both CTAs meet at a
// cluster barrier before tensor memory is freed.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "iq_fp4.cuh"
#include "iq_fp8.cuh"
#include "iq_internal.h"
#include "iq_ptx.cuh"

namespace iq {

__device__ uint32_t g_iq_status;

namespace {

constexpr int BM = 128;                          // token rows per CTA (256 per pair)
constexpr int BK = 128;
constexpr int kPair = 2;
constexpr uint16_t kPairMask = 0x3;
constexpr int kStages = 6;
static_assert(kNumKBlocks == 2 * kStages, "a tile is two passes over the ring (static phases in the MMA loop)");
constexpr int kABytes = BM * BK;                 // 16 KB: this CTA's token rows
constexpr int kNumEpiWarps = 8;
constexpr int kThreads = (2 + kNumEpiWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;                  // accumulators: columns 0..255
// Scale factors in tensor memory, two buffers (tile parity) so that a tile's
// copies are issued before the accumulator hand-off from the previous tile:
// SFA at kSfaCol + 32 b + 8 g (4 columns), SFB at kSfbCol + 32 b + 8 g + 4 h.
constexpr uint32_t kSfaCol = 256;
constexpr uint32_t kSfbCol = 320;
constexpr uint32_t kSfBufCols = 32;
// Two-head tiles: the RoPE rotation's cos/sin of each CTA row, per head of the
// tile (64 columns each), reused by the next tiles on the same token rows.
constexpr uint32_t kRopeCol = kSfbCol + 2 * kSfBufCols;
constexpr int kSfaWords = kScaleGroups * 128;    // per buffer
constexpr int kOutHeadBytes = BM * 64;           // FP4 codes of one head of the CTA's rows
constexpr int kNumBars = 2 * kStages + 2 + 2 + 2 + 2 + 1;

// Tile width kBN (output features per pair tile): 256 = two heads, each CTA
// loading 128 W rows (one head) per K-block; 128 = one head, each CTA loading
// 64 of its rows.  The narrow tile halves the MMA work per tile, so small and
// mid-size token counts spread over more SMs, and its 128-column accumulator
// fits twice in tensor memory, so a tile's epilogue overlaps the next tile's
// MMAs; the wide tile reads each X K-block once for two heads, which halves
// the X traffic from L2 to the SMs per FLOP at large token counts.
template <int kBN>
struct K2Layout {
  static constexpr int kHeads = kBN / kHeadDim;              // heads per tile
  static constexpr int kBBytes = (kBN / kPair) * BK;         // this CTA's W rows per K-block
  static constexpr int kStageTx = kPair * (kABytes + kBBytes);   // bytes landing per stage, both CTAs
  static constexpr int kAccBufs = kBN == 128 ? 2 : 1;        // accumulators in tensor memory
  static constexpr int kSfbWords = kScaleGroups * kBN;       // per buffer
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffSfa = kOffB + kStages * kBBytes;
  static constexpr int kOffSfb = kOffSfa + 2 * kSfaWords * 4;
  static constexpr int kOffOut = kOffSfb + 2 * kSfbWords * 4;   // FP4 code staging: [heads][128 rows][64 B]
  static constexpr int kOffBar = kOffOut + kHeads * kOutHeadBytes;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;    // + alignment slack
  static_assert(kBN == 128 || kBN == 256, "tile width");
  static_assert(kOffB % 1024 == 0 && kBBytes % 1024 == 0 && kOffOut % 1024 == 0, "swizzled tiles");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kAccBufs * kBN <= static_cast<int>(kSfaCol), "accumulators below the scale columns");
  static_assert(kSfbCol + 2 * kSfBufCols <= kTmemCols && kSfaCol + 2 * kSfBufCols <= kSfbCol, "scale columns");
  static_assert(kBN == 128 || kRopeCol + 64 * kHeads <= kTmemCols, "cos/sin columns");
};

__device__ __forceinline__ void fail(volatile uint32_t* abort_flag, uint32_t bit) {
  atomicOr(&g_iq_status, bit);
  *abort_flag = 1u;
}

// Progress flags of the fused quantizer, in the caller's workspace: word 0
// holds the call epoch E, word 1 + c the progress of CTA c as
// (tag(E, c) << 16) | k, k = the number of waves whose token rows the CTA has
// written (kExited once all of its threads are done).  Each CTA writes only
// its own word (plain release stores: no atomics, no contention), and a
// reader accepts a word only if it carries the tag of this call's epoch and
// that CTA, a 48-bit hash: a word left by an earlier call (another epoch) or
// anything a fresh workspace holds matches only by a 2^-48 chance, so no word
// needs clearing.  CTA 0 finishes last (it waits for every other CTA's exit
// flag) and then advances the epoch for the next call.
constexpr uint32_t kExited = 0xFFFFu;

// SplitMix64's finaliser (Steele, Lea and Flood, "Fast splittable
// pseudorandom number generators") over the epoch and the CTA index.
__device__ __forceinline__ uint64_t flag_tag(uint64_t epoch, uint32_t cta) {
  uint64_t z = epoch + 0x9E3779B97F4A7C15ull * (static_cast<uint64_t>(cta) + 1ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z >> 16;
}

__device__ __forceinline__ bool flag_reached(uint64_t word, uint64_t tag, uint32_t k) {
  return (word >> 16) == tag && (word & 0xFFFFull) >= k;
}

// Wave v of the interleaved order (tiles [vP, vP + P), one per pair) and the
// rows it reaches first: the 256-row blocks [blk_lo, blk_hi], rows [r0, r1).
struct WaveRows {
  int r0, r1;
  long long units;   // 3 per row: (row, group of four 128-blocks)
};
__device__ __forceinline__ WaveRows wave_rows(int v, int P, int T, int M, int tiles_per_row_block) {
  const int blk_hi = min(v * P + P - 1, T - 1) / tiles_per_row_block;
  const int blk_lo = v == 0 ? 0 : min(v * P - 1, T - 1) / tiles_per_row_block + 1;
  WaveRows w;
  w.r0 = blk_lo * 256;
  w.r1 = min((blk_hi + 1) * 256, M);
  w.units = w.r1 > w.r0 ? 3LL * (w.r1 - w.r0) : 0LL;
  return w;
}

// The CTA whose contiguous share [U c / G, U (c + 1) / G) of a wave's U units
// holds unit u.
__device__ __forceinline__ int unit_owner(long long u, long long units, int G) {
  return static_cast<int>(((u + 1) * G - 1) / units);
}

// NeoX RoPE on dims 0..63 of a (token, head): pairs (i, i+32), angle = pos *
// 10000^(-i/32).  The angle is reduced in turns with a two-float product
// (head and tail of the frequency, exact FMA residue) so that it stays
// accurate for large positions; the reduced angle lies in [-pi, pi].
// Frequencies i and i+1 go through the packed lanes together; rounding to an
// integer uses the 1.5 * 2^23 shift, exact for |turns| < 2^22.
//
// rope_cs_fill computes one row's cos/sin and keeps them in tensor memory at
// column taddr (this warp's lanes): frequency pair j = (2j, 2j+1) at columns
// 4j..4j+3 as (cos, cos, sin, sin).  Warp-collective: every lane of the warp
// takes part.
__device__ __forceinline__ void rope_cs_fill(int pos, const GemmArgs& args, uint32_t taddr) {
  const float pf = static_cast<float>(pos);
  const uint64_t pp = f2_pack(pf, pf);
  const uint64_t shift = f2_pack(12582912.0f, 12582912.0f);
  const uint64_t two_pi = f2_pack(kTwoPi, kTwoPi);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const uint64_t hi = f2_pack(args.rope.hi[i], args.rope.hi[i + 1]);
    const uint64_t lo = f2_pack(args.rope.lo[i], args.rope.lo[i + 1]);
    const uint64_t th = f2_mul(pp, hi);
    uint64_t tl = f2_fma(pp, hi, f2_neg(th));
    tl = f2_fma(pp, lo, tl);
    const uint64_t rn = f2_sub(f2_add(th, shift), shift);
    const uint64_t ang = f2_mul(f2_add(f2_sub(th, rn), tl), two_pi);
    float a0, a1, s0, c0, s1, c1;
    f2_unpack(ang, a0, a1);
    __sincosf(a0, &s0, &c0);
    __sincosf(a1, &s1, &c1);
    tmem_st_32x32b_x4(taddr + 2u * static_cast<uint32_t>(i), c0, c1, s0, s1);
  }
  tmem_st_wait();
}

// RoPE on p[0..31] (p[j] = dims 2j, 2j+1 as one packed pair) with the
// cos/sin that rope_cs_fill stored.  Warp-collective.
__device__ __forceinline__ void rope_apply_cached(uint64_t* p, uint32_t taddr) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float v[16];
    tmem_ld_32x32b_x16(taddr + 16u * static_cast<uint32_t>(q), v);
    tmem_ld_wait16(v);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int i = 2 * (4 * q + jj);
      const uint64_t c = f2_pack(v[4 * jj], v[4 * jj + 1]);
      const uint64_t s = f2_pack(v[4 * jj + 2], v[4 * jj + 3]);
      const uint64_t x1 = p[i >> 1], x2 = p[(i >> 1) + 16];
      p[i >> 1] = f2_fma(x1, c, f2_mul(x2, f2_neg(s)));        // x1 c - x2 s
      p[(i >> 1) + 16] = f2_fma(x2, c, f2_mul(x1, s));         // x2 c + x1 s
    }
  }
}

// Unscaled fast Walsh-Hadamard stages in Sylvester order over the 2 kN dims
// held in p[0..kN) (dim bits 0 .. log2(2 kN) - 1, lowest bit first).  The
// stage pairing dims that differ in bit 0 works inside each packed pair:
// (a, b) -> (a + b, a - b) = (a, b) * (1, -1) + (b, a).
template <int kN>
__device__ __forceinline__ void fwht_packed(uint64_t* p) {
  const uint64_t one_neg = f2_pack(1.0f, -1.0f);
#pragma unroll
  for (int j = 0; j < kN; ++j) {
    float a, b;
    f2_unpack(p[j], a, b);
    p[j] = f2_fma(p[j], one_neg, f2_pack(b, a));
  }
#pragma unroll
  for (int h = 1; h < kN; h <<= 1) {
#pragma unroll
    for (int j = 0; j < kN; ++j) {
      if ((j & h) == 0) {
        const uint64_t a = p[j], b = p[j + h];
        p[j] = f2_add(a, b);
        p[j + h] = f2_sub(a, b);
      }
    }
  }
}

// FP4 of z = v / sqrt(128) for the 2 kN Hadamard outputs in p[0..kN), whole
// blocks of the variant.  The codes of dims 32t..32t+31 (four words, word w
// = dims 8w..8w+7 as E2M1 nibbles) go to chunk(t, words) as soon as they are
// formed, so that few code registers are live; byte b of the result is block
// b's scale.
template <int kFmt, int kN, typename Chunk>
__device__ __forceinline__ uint64_t fp4_blocks(const uint64_t* p, Chunk&& chunk) {
  uint64_t sfb = 0;
  if constexpr (kFmt != kFp4Nv) {
    // MXFP4: per 32-block UE8M0 exponent e; codes = E2M1(z * 2^-e), formed
    // as v * (2^-e / sqrt(128)), equal to fp32(z) * 2^-e.
#pragma unroll
    for (int b = 0; b < kN / 16; ++b) {
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float x0, x1;
        f2_unpack(p[16 * b + j], x0, x1);
        amax = fmaxf(amax, fmaxf(fabsf(x0), fabsf(x1)));
      }
      const int e = fp4_block_exponent<kFmt>(amax * kInvSqrt128);
      const float k = fp4_code_factor(e);
      const uint64_t kk = f2_pack(k, k);
      uint32_t codes[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        float q[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) f2_unpack(f2_mul(p[16 * b + 4 * t + j], kk), q[2 * j], q[2 * j + 1]);
        codes[t] = cvt_e2m1x8(q);
      }
      chunk(b, codes);
      sfb |= static_cast<uint64_t>(e + 127) << (8 * b);
    }
  } else {
    // NVFP4-style: per 16-block E4M3 scale s = E4M3(max(amax_z, 1e-4) / 6);
    // codes = E2M1(v * (1/s) / sqrt(128)).  Two blocks at a time in packed
    // arithmetic; the reciprocal comes from the scale's code (no division).
    const uint64_t c2 = f2_pack(kInvSqrt128, kInvSqrt128);
    const uint64_t sixth = f2_pack(kSixth, kSixth);
#pragma unroll
    for (int b = 0; b < kN / 8; b += 2) {
      float am[2] = {0.f, 0.f};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float x0, x1;
          f2_unpack(p[8 * (b + h) + j], x0, x1);
          am[h] = fmaxf(am[h], fmaxf(fabsf(x0), fabsf(x1)));
        }
      }
      float z0, z1;
      f2_unpack(f2_mul(f2_pack(am[0], am[1]), c2), z0, z1);
      float t0, t1;
      f2_unpack(f2_mul(f2_pack(fmaxf(z0, kAmaxFloor), fmaxf(z1, kAmaxFloor)), sixth), t0, t1);
      const uint32_t code0 = nvfp4_code(t0), code1 = nvfp4_code(t1);
      float k0, k1;
      f2_unpack(f2_mul(f2_pack(e4m3_reciprocal(code0), e4m3_reciprocal(code1)), c2), k0, k1);
      uint32_t codes[4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float kh = h == 0 ? k0 : k1;
        const uint64_t kk = f2_pack(kh, kh);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          float q[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) f2_unpack(f2_mul(p[8 * (b + h) + 4 * t + j], kk), q[2 * j], q[2 * j + 1]);
          codes[2 * h + t] = cvt_e2m1x8(q);
        }
      }
      chunk(b / 2, codes);
      sfb |= static_cast<uint64_t>(code0 | (code1 << 8)) << (8 * b);
    }
  }
  return sfb;
}

// FP4 codes, scales and the optional pre-quant output of dims
// [128 kN/64 * part, +2 kN) of one (token, head), from its Hadamard outputs in
// p[0..kN): kN = 64 is the whole head (part 0), kN = 32 one half of it.  The
// codes go to `stage_row`, the (token, head)'s 64 bytes of the shared staging
// tile, stored with the 64-byte swizzle of the bulk tensor store (16-byte
// chunk c of row r at chunk c ^ ((r >> 1) & 3)): a warp's 16-byte writes then
// fall on distinct banks.
template <int kFmt, int kN>
__device__ __forceinline__ void fp4_store(const uint64_t* p, int row, int head, int part, const GemmArgs& args,
                                          uint8_t* stage_row, int swz) {
  using F = Fp4Layout<kFmt>;
  constexpr int kBlocks = 2 * kN / F::kBlock;    // scale bytes this call writes
  constexpr int kChunks = kN / 16;               // 16-byte code chunks
  const uint64_t sfb = fp4_blocks<kFmt, kN>(p, [&](int t, const uint32_t (&c)[4]) {
    *reinterpret_cast<uint4*>(stage_row + (((part * kChunks + t) ^ swz) << 4)) = make_uint4(c[0], c[1], c[2], c[3]);
  });
  uint8_t* sf = args.q_sf + static_cast<long long>(row) * F::kScaleBytesPerToken + head * F::kBlocksPerHead +
                part * kBlocks;
  if constexpr (kBlocks == 8) {
    *reinterpret_cast<uint2*>(sf) = make_uint2(static_cast<uint32_t>(sfb), static_cast<uint32_t>(sfb >> 32));
  } else if constexpr (kBlocks == 4) {
    *reinterpret_cast<uint32_t*>(sf) = static_cast<uint32_t>(sfb);
  } else {
    static_assert(kBlocks == 2, "scale bytes per call");
    *reinterpret_cast<uint16_t*>(sf) = static_cast<uint16_t>(sfb);
  }
  if (args.q_pre != nullptr) {
    const uint64_t c2 = f2_pack(kInvSqrt128, kInvSqrt128);
    float4* pre = reinterpret_cast<float4*>(args.q_pre + static_cast<long long>(row) * kQDim + head * kHeadDim +
                                            part * 2 * kN);
#pragma unroll
    for (int t = 0; t < kN / 2; ++t) {
      float z0, z1, z2, z3;
      f2_unpack(f2_mul(p[2 * t], c2), z0, z1);
      f2_unpack(f2_mul(p[2 * t + 1], c2), z2, z3);
      pre[t] = make_float4(z0, z1, z2, z3);
    }
  }
}

// kNoLoads: the wait self-test instance.  Its producer issues no TMA loads,
// so the stage barriers the MMA issuer waits on never complete, no MMA is
// issued, and the MMA issuer's, the epilogue's and the producer's bounded
// waits all give up with nothing asynchronous in flight (the only tensor-core
// work is the scale-factor copy, which completes).  It exercises the give-up
// and teardown path; the product launches only kNoLoads = false.
template <int kFmt, int kBN, bool kNoLoads = false, bool kFuse = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_rope_hadamard_fp4_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                                  const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ GemmArgs args) {
  static_assert(!kFuse || (kBN == 256 && !kNoLoads), "the fused quantizer runs with two-head tiles");
  // The next kernel of the stream may be scheduled as soon as every CTA of
  // this one runs: the quantizer of the next call, for instance, then starts
  // while this kernel works and waits for its completion before it touches
  // memory.
  grid_launch_dependents();
  using L = K2Layout<kBN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem + L::kOffA;
  uint8_t* sB = smem + L::kOffB;
  uint32_t* sSfa = reinterpret_cast<uint32_t*>(smem + L::kOffSfa);
  uint32_t* sSfb = reinterpret_cast<uint32_t*>(smem + L::kOffSfb);
  uint8_t* sOut = smem + L::kOffOut;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* full = bars;                       // leader: both CTAs' loads of a stage landed
  uint64_t* empty = bars + kStages;            // both: the pair's MMAs released a stage
  uint64_t* sf_full = bars + 2 * kStages;      // leader: both CTAs staged a tile's scales
  uint64_t* sf_empty = sf_full + 2;            // both: the scale copies completed
  uint64_t* tmem_full = sf_empty + 2;          // both: accumulator b holds a complete tile
  uint64_t* tmem_empty = tmem_full + 2;        // leader: both CTAs drained accumulator b
  uint64_t* final_bar = tmem_empty + 2;        // both: every pair MMA has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t timeout = args.timeout_ns;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  // Epilogue warps that read the accumulator: four per head of the tile (one
  // per 32-lane quarter of tensor memory).
  constexpr int kDrainWarps = kNumEpiWarps;    // every epilogue warp drains every tile

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_q);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sf_full[b], kPair);
      mbar_init(&sf_empty[b], 1);
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], kPair * kDrainWarps);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  // Barriers and tensor memory must be ready in both CTAs before either
  // issues anything that touches the other.
  tc_fence_before_sync();
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // Fused quantizer: this call's epoch (CTA 0 advances it only after every
  // CTA has flagged its exit, so all CTAs read the same value).
  [[maybe_unused]] uint64_t epoch = 0;
  if constexpr (kFuse) epoch = *reinterpret_cast<const volatile unsigned long long*>(args.ready);

  // Leader-CTA addresses of the barriers that collect the pair's work.
  const uint32_t full_leader0 = mapa_shared(smem_u32(&full[0]), 0);
  const uint32_t sf_full_leader0 = mapa_shared(smem_u32(&sf_full[0]), 0);
  const uint32_t tmem_empty_leader0 = mapa_shared(smem_u32(&tmem_empty[0]), 0);

  // Pair tile pt covers token rows [256 mp, +256) (split by CTA rank) and
  // features [kBN n, +kBN).  In feature-major order (mp = pt % num_m_pairs)
  // consecutive tiles share their heads; in token-major order (mp = pt /
  // n_tiles, the default) they share their token rows, so the pairs running
  // at one time read few distinct X row blocks, each from HBM once, while W
  // (12.6 MB) stays in L2.  A pair takes a contiguous run of tiles, or, in
  // the interleaved order, tiles p, p + P, p + 2P, ... (P pairs), so that the
  // pairs' i-th tiles together form the i-th run of P consecutive tiles.
  constexpr int n_tiles = kQDim / kBN;
  const int num_pairs = static_cast<int>(cluster_count_x());
  const int pair_id = static_cast<int>(cluster_id_x());
  const bool interleaved = args.order == kOrderInterleaved;
  int my_first, my_step, my_count;
  if (interleaved) {
    my_first = pair_id;
    my_step = num_pairs;
    my_count = pair_id < args.num_pair_tiles ? (args.num_pair_tiles - 1 - pair_id) / num_pairs + 1 : 0;
  } else {
    const int tiles_per_pair = (args.num_pair_tiles + num_pairs - 1) / num_pairs;
    my_first = pair_id * tiles_per_pair;
    my_step = 1;
    my_count = max(0, min(tiles_per_pair, args.num_pair_tiles - my_first));
  }
  auto tile_at = [&](int i) { return my_first + i * my_step; };
  const int num_m_pairs = args.num_m_pairs;
  const bool token_major = args.order != kOrderFeatureMajor;
  auto tile_mp = [&](int pt) { return token_major ? pt / n_tiles : pt % num_m_pairs; };
  auto tile_n = [&](int pt) { return token_major ? pt % n_tiles : pt / num_m_pairs; };
  auto tile_m0 = [&](int pt) { return (tile_mp(pt) * kPair + static_cast<int>(rank)) * BM; };

  // The producer's first tile: W and its scales are inputs the preceding
  // kernel does not write (the quantizer writes only the FP8 latent and its
  // scales), so the first pass of W loads over the ring and the first
  // weight-scale words are issued before the dependency wait and overlap
  // that kernel.  The stages are fresh, so no release wait precedes them; the
  // leader's expected byte count covers the X loads issued after the wait.
  uint32_t rb[kScaleGroups][L::kHeads];   // producer: the tile's heads' weight-scale words per group
  auto fetch_w_scales = [&](int i) {
    if (i >= my_count) return;
    const int n_tile = tile_n(tile_at(i));
#pragma unroll
    for (int g = 0; g < kScaleGroups; ++g) {
#pragma unroll
      for (int h = 0; h < L::kHeads; ++h) {
        const uint8_t* ws = args.w_sf + (n_tile * L::kHeads + h) * kNumKBlocks + 4 * g;
        rb[g][h] = static_cast<uint32_t>(__ldg(ws)) | (static_cast<uint32_t>(__ldg(ws + 1)) << 8) |
                   (static_cast<uint32_t>(__ldg(ws + 2)) << 16) | (static_cast<uint32_t>(__ldg(ws + 3)) << 24);
      }
    }
  };
  const bool have_tile = my_count > 0;
  // Set by the epilogue warps once they have arrived on the final cluster
  // barrier (right after their last accumulator read).
  bool cluster_arrived = false;
  if (warp == 0) {
    if constexpr (!kNoLoads) {
      if (lane == 0 && have_tile) {
        const int n0 = tile_n(tile_at(0)) * kBN + static_cast<int>(rank) * (kBN / kPair);
        for (int kb = 0; kb < kStages; ++kb) {
          if (leader) mbar_arrive_expect_tx(&full[kb], L::kStageTx);
          tma_load_2d_pair(sB + kb * L::kBBytes, &tm_w, full_leader0 + 8u * kb, kb * BK, n0);
        }
      }
    }
    fetch_w_scales(0);
  }
  // Launched with programmatic stream serialization: everything above
  // overlapped the preceding kernel; nothing below runs before it completed
  // (apart from the W loads and weight-scale reads above, no global memory is
  // read or written before this point).
  grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0;
    uint32_t issued_mask = 0, issued_phase = 0;   // per stage: a load was issued / its phase
    // Fused quantizer: before it reads a tile's token rows (FP8 codes by TMA,
    // scale words by plain loads) the producer waits until the block's
    // counter shows all of its units written (3 per row), acquires it, and
    // orders the async proxy behind it.  All lanes take part.
    auto rows_ready = [&](int i) -> bool {
      if constexpr (!kFuse) {
        return true;
      } else {
        if (i >= my_count) return true;
        const int pt = tile_at(i);
        const int m0 = tile_m0(pt);
        const int rows = min(BM, args.M - m0);
        if (rows <= 0) return true;   // rows past M: the loads read zeros
        // The wave that first reaches this row block, and the CTAs whose
        // shares of that wave hold the block's units.
        const int v = (tile_mp(pt) * n_tiles) / num_pairs;
        const WaveRows w = wave_rows(v, num_pairs, args.num_pair_tiles, args.M, n_tiles);
        const long long u0 = 3LL * (m0 - w.r0), u1 = u0 + 3LL * rows;
        const int G = static_cast<int>(gridDim.x);
        const int c_lo = unit_owner(u0, w.units, G), c_hi = unit_owner(u1 - 1, w.units, G);
        const uint32_t need = static_cast<uint32_t>(v + 1);
        bool ok = true;
        for (int c = c_lo + lane; c <= c_hi && ok; c += 32) {
          const uint64_t tag = flag_tag(epoch, static_cast<uint32_t>(c));
          const unsigned long long* f = args.ready + 1 + c;
          if (!flag_reached(ld_acquire_u64(f), tag, need)) {
            const uint64_t t0 = globaltimer_ns();
            while (true) {
              __nanosleep(32);
              if (flag_reached(ld_acquire_u64(f), tag, need)) break;
              if (globaltimer_ns() - t0 > timeout) {
                ok = false;
                break;
              }
            }
          }
        }
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (ok) fence_proxy_async_global();
        return ok;
      }
    };
    if constexpr (kFuse) {
      // The first tile's X loads go out whatever the outcome, so that every
      // stage whose W half is in flight completes.
      if (have_tile && !rows_ready(0) && lane == 0) fail(abort_flag, kStatusRowsWait);
    }
    // The first tile's X loads of the first pass go out at once (their W
    // halves are already in flight), ahead of the scale-word reads.
    if constexpr (!kNoLoads) {
      if (lane == 0 && have_tile) {
        const int m0 = tile_m0(tile_at(0));
        for (int kb = 0; kb < kStages; ++kb)
          tma_load_2d_pair(sA + kb * kABytes, &tm_x, full_leader0 + 8u * kb, kb * BK, m0);
        issued_mask = (1u << kStages) - 1u;
        issued_phase = 0u;
        phase = 1;
      }
    }
    // The next tile's scale words are fetched into registers while the
    // current tile's K-blocks stream, so no global-load latency sits at a
    // tile boundary.  ra: this lane's 4 rows x 3 groups of activation-scale
    // words (written by the preceding kernel: read after the wait).
    uint32_t ra[kScaleGroups][4];
    auto fetch_x_scales = [&](int i) {
      if (i >= my_count) return;
      const int m0 = tile_m0(tile_at(i));
#pragma unroll
      for (int g = 0; g < kScaleGroups; ++g) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int m = m0 + c * 32 + lane;
          ra[g][c] = m < args.m_al ? ld_dependent_u32(args.x_sf + static_cast<long long>(g) * args.m_al + m) : 0u;
        }
      }
    };
    fetch_x_scales(0);
    for (int local = 0; local < my_count; ++local) {
      // Every exit decision is made warp-uniform: the lanes must stay
      // converged for the shuffles below.
      if (__any_sync(0xFFFFFFFFu, *abort_flag != 0u)) break;
      const int pt = tile_at(local);
      const int m0 = tile_m0(pt);
      const int n_tile = tile_n(pt);
      const int buf = local & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sf_empty[buf], ((local >> 1) & 1) ^ 1, timeout))) {
        if (lane == 0) fail(abort_flag, kStatusProducerWait);
        break;
      }
      // Scale factors in the tcgen05.cp 32x128b layout: word [r * 4 + c] of a
      // 128-row tile holds row c * 32 + r.  SFA: this CTA's 128 token rows;
      // SFB: the tile's heads (128 rows each, all of them in both CTAs).
      uint32_t* sfa = sSfa + buf * kSfaWords;
      uint32_t* sfb = sSfb + buf * L::kSfbWords;
#pragma unroll
      for (int g = 0; g < kScaleGroups; ++g) {
        *reinterpret_cast<uint4*>(sfa + g * 128 + lane * 4) = make_uint4(ra[g][0], ra[g][1], ra[g][2], ra[g][3]);
#pragma unroll
        for (int h = 0; h < L::kHeads; ++h)
          *reinterpret_cast<uint4*>(sfb + g * kBN + h * 128 + lane * 4) =
              make_uint4(rb[g][h], rb[g][h], rb[g][h], rb[g][h]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if constexpr (!kFuse) {
        fetch_x_scales(local + 1);
        fetch_w_scales(local + 1);
      }
      bool ok = true;
      if (lane == 0) {
        mbar_arrive_cluster(sf_full_leader0 + 8u * static_cast<uint32_t>(buf));
        for (int kb = (local == 0 && !kNoLoads) ? kStages : 0; kb < kNumKBlocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, timeout)) {
            fail(abort_flag, kStatusProducerWait);
            ok = false;
            break;
          }
          if constexpr (!kNoLoads) {
            if (leader) mbar_arrive_expect_tx(&full[stage], L::kStageTx);
            const uint32_t bar = full_leader0 + 8u * stage;
            tma_load_2d_pair(sA + stage * kABytes, &tm_x, bar, kb * BK, m0);
            tma_load_2d_pair(sB + stage * L::kBBytes, &tm_w, bar, kb * BK,
                             n_tile * kBN + static_cast<int>(rank) * (kBN / kPair));
            issued_mask |= 1u << stage;
            issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      if constexpr (kFuse) {
        // After this tile's loads, so that a wait for the next tile's rows
        // never holds them back; the scale reads overlap the tile's last
        // MMAs.
        fetch_w_scales(local + 1);
        if (!rows_ready(local + 1)) {
          if (lane == 0) fail(abort_flag, kStatusRowsWait);
          break;
        }
        fetch_x_scales(local + 1);
      }
    }
    // Teardown: this CTA's loads signal the leader's barriers, so their
    // landing is observed through the stage's release by the pair's MMAs,
    // which consumed them.  The teardown waits get twice the limit (see the
    // final-commit wait below).
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        if ((issued_mask >> s) & 1u) {
          if (!mbar_wait(&empty[s], (issued_phase >> s) & 1u, 2 * timeout)) fail(abort_flag, kStatusTeardownWait);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------- MMA issuer (leader)
    if (lane == 0) {
      if (leader) {
        bool ok = true;
        const uint64_t adesc0 = smem_desc_sw128(smem_u32(sA));
        const uint64_t bdesc0 = smem_desc_sw128(smem_u32(sB));
        const uint32_t idesc0 = idesc_mxf8_e4m3(kPair * BM, kBN, 0, 0);
        for (int local = 0; local < my_count && ok; ++local) {
          if (*abort_flag) break;
          const int buf = local & 1;
          const int acc = local % L::kAccBufs;
          // The scale factors of this tile go to TMEM buffer `buf`, last read by
          // the tile two before, which is complete once that tile's
          // accumulator was drained: with one accumulator that was waited for
          // at the previous tile, so the copies are issued before this tile's
          // accumulator wait (off the hand-off); with two, after it.
          const uint32_t sfa_col = kSfaCol + kSfBufCols * static_cast<uint32_t>(buf);
          const uint32_t sfb_col = kSfbCol + kSfBufCols * static_cast<uint32_t>(buf);
          auto copy_scales = [&]() {
            tc_fence_after_sync();
            const uint32_t* sfa = sSfa + buf * kSfaWords;
            const uint32_t* sfb = sSfb + buf * L::kSfbWords;
#pragma unroll
            for (int g = 0; g < kScaleGroups; ++g) {
              tc_cp_32x128b_warpx4_pair(tmem + sfa_col + 8 * g, smem_desc_sf(smem_u32(sfa + g * 128)));
#pragma unroll
              for (int h = 0; h < L::kHeads; ++h)
                tc_cp_32x128b_warpx4_pair(tmem + sfb_col + 8 * g + 4 * h,
                                          smem_desc_sf(smem_u32(sfb + g * kBN + h * 128)));
            }
            tc_commit_pair(&sf_empty[buf], kPairMask);
          };
          if (!mbar_wait(&sf_full[buf], (local >> 1) & 1, timeout)) {
            fail(abort_flag, kStatusMmaWait);
            break;
          }
          if constexpr (L::kAccBufs == 1) copy_scales();
          if (!mbar_wait(&tmem_empty[acc], ((local / L::kAccBufs) & 1) ^ 1, timeout)) {
            fail(abort_flag, kStatusMmaWait);
            break;
          }
          tc_fence_after_sync();
          if constexpr (L::kAccBufs == 2) copy_scales();
          const uint32_t d_tmem = tmem + kAccCol + static_cast<uint32_t>(acc * kBN);
          // The K loop does little between MMAs: a tile is exactly two
          // passes over the ring, so every stage index, barrier phase, scale
          // ID and descriptor offset below is a compile-time constant and the
          // issuing thread spends few instructions per stage (it shares its
          // scheduler with two epilogue warps).  TMA data needs no tcgen05
          // fence: the barrier's transaction completion orders it.
#pragma unroll
          for (int kb = 0; kb < kNumKBlocks; ++kb) {
            const int s = kb % kStages;
            if (!mbar_wait(&full[s], static_cast<uint32_t>(kb / kStages) & 1u, timeout)) {
              fail(abort_flag, kStatusMmaWait);
              ok = false;
              break;
            }
            const uint64_t adesc = adesc0 + static_cast<uint64_t>(s * (kABytes >> 4));
            const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(s * (L::kBBytes >> 4));
            const uint32_t sfid = static_cast<uint32_t>(kb & 3);
            const uint32_t idesc = idesc0 | (sfid << 4) | (sfid << 29);
            const uint32_t sf_off = 8u * static_cast<uint32_t>(kb >> 2);
#pragma unroll
            for (int k = 0; k < BK / 32; ++k) {
              // advance 32 bytes along K inside the 128-byte swizzle atom
              tc_mma_mxf8_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, tmem + sfa_col + sf_off,
                               tmem + sfb_col + sf_off, (kb | k) != 0);
            }
            tc_commit_pair(&empty[s], kPairMask);   // frees the stage in both CTAs
          }
          if (ok) tc_commit_pair(&tmem_full[acc], kPairMask);
        }
        tc_commit_pair(final_bar, kPairMask);
      }
      // Teardown (both CTAs): every pair MMA writing this CTA's tensor memory
      // or reading its shared memory has completed.  The teardown waits get
      // twice the limit: the other CTA's issuer reaches its final commit only
      // after its own waits, each of which may use the whole limit before it
      // gives up.
      if (!mbar_wait(final_bar, 0, 2 * timeout)) fail(abort_flag, kStatusTeardownWait);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;            // the TMEM lane group this warp may read
    // Two-head tiles: warps 2-5 take the first head, 6-9 the second.  One-head
    // tiles: warps w and w + 4 (the same TMEM lanes) share each (token, head),
    // w the Hadamard outputs 0..63 and w + 4 the outputs 64..127.
    const int half = (warp - 2) >> 2;
    const int trow = quad * 32 + lane;    // row within the CTA's 128-row tile
    uint8_t* stage_row = sOut + (L::kHeads == 2 ? half : 0) * kOutHeadBytes + trow * 64;
    const int swz = (trow >> 1) & 3;
    const bool store_issuer = warp == 2 && lane == 0;
    // Fused quantizer.  Wave v of the interleaved order is the run of tiles
    // [vP, vP + P), one per pair, and a pair's i-th tile lies in wave i.  The
    // wave's new rows are the 256-row blocks that no earlier wave reaches;
    // their units (row, group of four 128-blocks) are split into G equal
    // contiguous ranges, one per CTA, and dealt round-robin to its eight
    // epilogue warps.  A producer needs wave i + 1's rows when its MMAs are
    // half way through tile i (the ring runs half a tile ahead), so the warps
    // quantize waves 0, 1 and 2 before the first accumulator wait and wave
    // i + 2 before the wait for tile i, after tile i - 1's epilogue: at least
    // half a tile of slack.  After its share of a wave the CTA publishes the
    // number of waves it has done in its progress flag.
    [[maybe_unused]] int q_next = 0;
    [[maybe_unused]] const int num_waves = (args.num_pair_tiles + num_pairs - 1) / num_pairs;
    auto quantize_wave = [&](int v) {
      const WaveRows w = wave_rows(v, num_pairs, args.num_pair_tiles, args.M, n_tiles);
      const int r0 = w.r0;
      const long long units = w.units;
      const long long G = gridDim.x;
      const long long lo = units * blockIdx.x / G, hi = units * (blockIdx.x + 1) / G;
      const int ew = warp - 2;
      auto unit_src = [&](long long u) {
        return args.latent + static_cast<long long>(r0 + static_cast<int>(u / 3)) * kLatentDim +
               static_cast<int>(u % 3) * 512 + lane * 16;
      };
      auto unit_store = [&](long long u, const uint4& a, const uint4& b) {
        const int row = r0 + static_cast<int>(u / 3);
        const int g = static_cast<int>(u % 3);
        uint4 codes;
        const uint32_t word = fp8_quant_unit(a, b, true, codes);
        *reinterpret_cast<uint4*>(args.x_fp8 + static_cast<long long>(row) * kLatentDim + g * 512 + lane * 16) = codes;
        if (lane == 0) {
          int32_t* sf = args.x_sf_out + static_cast<long long>(g) * args.m_al;
          sf[row] = static_cast<int32_t>(word);
          if (row == args.M - 1)
            for (int r = args.M; r < args.m_al; ++r) sf[r] = 0;   // pad rows, as the quantizer kernel writes them
        }
      };
      // Two units per warp in flight: both loads go out before either unit
      // is reduced.
      for (long long u = lo + ew; u < hi; u += 2 * kNumEpiWarps) {
        const long long u2 = u + kNumEpiWarps;
        const bool two = u2 < hi;   // warp-uniform
        const uint16_t* s1 = unit_src(u);
        const uint4 a1 = ld_stream_v4(s1), b1 = ld_stream_v4(s1 + 8);
        uint4 a2 = make_uint4(0, 0, 0, 0), b2 = a2;
        if (two) {
          const uint16_t* s2 = unit_src(u2);
          a2 = ld_stream_v4(s2);
          b2 = ld_stream_v4(s2 + 8);
        }
        unit_store(u, a1, b1);
        if (two) unit_store(u2, a2, b2);
      }
      if (args.quant_delay_ns != 0ull && lane == 0) {
        // Diagnostics only: holds back the wave's signal (bounded by the delay).
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < args.quant_delay_ns) {
        }
      }
      // The warps meet, then one thread publishes the CTA's progress with a
      // release (cumulative over the other threads' stores, which the
      // barrier ordered before it).
      named_barrier_sync(1, kNumEpiWarps * 32);
      if (ew == 0 && lane == 0) {
        __threadfence();
        st_release_u64(args.ready + 1 + blockIdx.x,
                       (flag_tag(epoch, blockIdx.x) << 16) | static_cast<uint64_t>(v + 1));
      }
    };
    // One tile ahead of its quantization, the CTA's share of a wave's token
    // rows is fetched from HBM into L2 (asynchronous bulk prefetches, one per
    // 1 KB unit), so that the warps' loads later hit L2.
    auto prefetch_wave = [&](int v) {
      if constexpr (kFuse) {
        if (v >= num_waves) return;
        const WaveRows w = wave_rows(v, num_pairs, args.num_pair_tiles, args.M, n_tiles);
        const long long G = gridDim.x;
        const long long lo = w.units * blockIdx.x / G, hi = w.units * (blockIdx.x + 1) / G;
        for (long long u = lo + (warp - 2) * 32 + lane; u < hi; u += kNumEpiWarps * 32) {
          const uint16_t* src = args.latent + static_cast<long long>(w.r0 + static_cast<int>(u / 3)) * kLatentDim +
                                static_cast<int>(u % 3) * 512;
          prefetch_l2_bulk(src, 1024);
        }
      }
    };
    auto quantize_through = [&](int v_last) {
      if constexpr (kFuse) {
        for (; q_next <= v_last && q_next < num_waves; ++q_next) quantize_wave(q_next);
        prefetch_wave(q_next);
      }
    };
    int rope_mp = -1;   // the row block whose cos/sin are in tensor memory
    for (int local = 0; local < my_count; ++local) {
      quantize_through(local + 2);
      const int pt = tile_at(local);
      const bool rope_cached = tile_mp(pt) == rope_mp;   // warp-uniform
      rope_mp = tile_mp(pt);
      const int row = tile_m0(pt) + trow;
      const int head = tile_n(pt) * L::kHeads + (L::kHeads == 2 ? half : 0);
      const int acc = local % L::kAccBufs;
      const int pos = row < args.M ? static_cast<int>(ld_dependent_u32(args.pos + row)) : 0;   // in flight during the wait
      // The rotation's cos/sin depend on the row alone, so they are computed
      // while the tile's MMAs run (before the accumulator wait), only on a
      // pair's first tile of a row block, and read back from tensor memory
      // (one-head tiles: by the warps of dims 0..63 alone).
      const uint32_t rope_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + kRopeCol +
                                 static_cast<uint32_t>(L::kHeads == 2 ? 64 * half : 0);
      const bool rope_warp = L::kHeads == 2 || half == 0;   // warp-uniform
      if (rope_warp && !rope_cached) rope_cs_fill(pos, args, rope_addr);
      // The previous tile's bulk stores must have read the staging tile
      // before anyone overwrites it.
      if (store_issuer) tma_store_wait_read();
      const bool got = mbar_wait(&tmem_full[acc], (local / L::kAccBufs) & 1, timeout);
      if (!got) fail(abort_flag, kStatusEpilogueWait);
      // One decision for all epilogue warps (they meet at a named barrier
      // below); this barrier also tells them the staging tile is free.
      if (!named_barrier_and(1, kNumEpiWarps * 32, got && *abort_flag == 0u)) break;
      if constexpr (L::kHeads == 1) {
        // Sylvester's H_128 = H_2 (x) H_64: the outputs 64 h + i are
        // H_64(x_0)[i] + (-1)^h H_64(x_1)[i], x_0 = dims 0..63 after RoPE and
        // x_1 = dims 64..127.  Each warp transforms its own half in place in
        // tensor memory, the pair meets at a named barrier, and each reads
        // the other half back: the same operations on every element as in one
        // thread, so the bytes are the same.
        tc_fence_after_sync();
        float v[64];
        const uint32_t trow_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + kAccCol +
                                   static_cast<uint32_t>(acc * kBN);
        const uint32_t mine = trow_addr + static_cast<uint32_t>(64 * half);
        const uint32_t theirs = trow_addr + static_cast<uint32_t>(64 * (half ^ 1));
        tmem_ld_32x32b_x32(mine, v);
        tmem_ld_32x32b_x32(mine + 32, v + 32);
        tmem_ld_wait(v);
        tmem_ld_wait(v + 32);
        uint64_t p[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) p[j] = f2_pack(v[2 * j], v[2 * j + 1]);
        if (half == 0) rope_apply_cached(p, rope_addr);
        fwht_packed<32>(p);
#pragma unroll
        for (int j = 0; j < 32; ++j) f2_unpack(p[j], v[2 * j], v[2 * j + 1]);
        tmem_st_32x32b_x32(mine, v);
        tmem_st_32x32b_x32(mine + 32, v + 32);
        tmem_st_wait();
        tc_fence_before_sync();
        named_barrier_sync(2 + quad, 64);
        tc_fence_after_sync();
        tmem_ld_32x32b_x32(theirs, v);
        tmem_ld_32x32b_x32(theirs + 32, v + 32);
        tmem_ld_wait(v);
        tmem_ld_wait(v + 32);
        tc_fence_before_sync();
        __syncwarp();
        // The pair's last tile needs no release: nothing waits for it, and
        // without this remote arrive no cluster access of this CTA is left in
        // flight at the final cluster barrier (see there).
        if (lane == 0 && local != my_count - 1)
          mbar_arrive_remote(tmem_empty_leader0 + 8u * static_cast<uint32_t>(acc));
        if (!kFuse && local == my_count - 1) {
          cluster_arrive_relaxed();
          cluster_arrived = true;
        }
        // The last stage (dim bit 6): a + b in the first half, a - b in the
        // second, a being the first half's values.
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const uint64_t o = f2_pack(v[2 * j], v[2 * j + 1]);
          p[j] = half == 0 ? f2_add(p[j], o) : f2_sub(o, p[j]);
        }
        if (row < args.M) fp4_store<kFmt, 32>(p, row, head, half, args, stage_row, swz);
      } else {
        tc_fence_after_sync();
        float v[128];
        const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + kAccCol +
                               static_cast<uint32_t>(acc * kBN + half * 128);
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
        // The accumulator values are in registers (tcgen05.wait::ld above), so
        // the leader may overwrite it: a CTA-scope arrive suffices and does not
        // wait for earlier global stores to reach L2.
        if (lane == 0 && local != my_count - 1)   // none for the last tile (see the one-head path)
          mbar_arrive_remote(tmem_empty_leader0 + 8u * static_cast<uint32_t>(acc));
        uint64_t p[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) p[j] = f2_pack(v[2 * j], v[2 * j + 1]);
        rope_apply_cached(p, rope_addr);
        fwht_packed<64>(p);
        if (row < args.M) fp4_store<kFmt, 64>(p, row, head, 0, args, stage_row, swz);
      }
      fence_proxy_async_smem();
      named_barrier_sync(1, kNumEpiWarps * 32);
      if (store_issuer) {
        // Rows past M are clipped by the bulk store.
#pragma unroll
        for (int h = 0; h < L::kHeads; ++h)
          tma_store_2d(&tm_q, sOut + h * kOutHeadBytes, (tile_n(pt) * L::kHeads + h) * 64, tile_m0(pt));
        tma_store_commit();
      }
    }
    // A pair with fewer tiles than waves still owes its share of the rest.
    quantize_through(num_waves - 1);
    // The staging tile must stay valid until the last bulk stores have read
    // it; their writes to global memory complete with the grid.
    if (store_issuer) tma_store_wait_read();
  }

  // Neither CTA leaves (or frees tensor memory) while the pair may still use
  // its shared memory, barriers or tensor memory.  Every access of one CTA to
  // the other's shared memory has been seen to complete by then (loads and
  // MMAs through the stage and final barriers, scale-staging arrives through
  // the issuer's waits, accumulator releases through the issuer's waits, and
  // the last tile sends none), so the arrive publishes nothing and is
  // relaxed: a release arrive waited for this CTA's outstanding stores
  // (~0.2 us per call at 256 and 512 tokens).  With one-head tiles the
  // epilogue warps arrive as soon as their last accumulator read is done.
  // (With two-head tiles that early arrive, then a release, measured ~1 %
  // slower at 4632 tokens.)
  tc_fence_before_sync();
  if (!cluster_arrived) cluster_arrive_relaxed();
  cluster_wait();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
  if constexpr (kFuse) {
    // Every CTA flags its exit once all of its threads are done.  CTA 0 then
    // waits (bounded) for all the others, so that no CTA of this call can
    // still read the epoch, and advances it for the next call (also when the
    // wait gives up, so that a later call never meets this call's flags).
    if (threadIdx.x == 0) {
      __threadfence();
      st_release_u64(args.ready + 1 + blockIdx.x, (flag_tag(epoch, blockIdx.x) << 16) | kExited);
    }
    if (blockIdx.x == 0 && warp == 0) {
      // The 32 lanes poll the other CTAs' flags side by side.
      const uint64_t t0 = globaltimer_ns();
      bool ok = true;
      for (uint32_t c = 1 + lane; c < gridDim.x && ok; c += 32) {
        const uint64_t tag = flag_tag(epoch, c);
        while (!flag_reached(ld_acquire_u64(args.ready + 1 + c), tag, kExited)) {
          if (globaltimer_ns() - t0 > 2 * timeout) {
            ok = false;
            break;
          }
          __nanosleep(32);
        }
      }
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (lane == 0) {
        if (!ok) atomicOr(&g_iq_status, kStatusRowsWait);
        *reinterpret_cast<volatile unsigned long long*>(args.ready) = epoch + 1ull;
      }
    }
  }
}

// Cluster of two, plus programmatic stream serialization: the kernel may be
// scheduled while the preceding kernel of the stream (the quantizer) runs;
// it waits for that kernel's completion (griddepcontrol.wait) before any
// global memory access.
cudaLaunchConfig_t pair_config(int pairs, int smem_bytes, cudaLaunchAttribute* attr, cudaStream_t stream) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pairs * kPair, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

template <int kFmt, int kBN, bool kNoLoads = false, bool kFuse = false>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(gemm_rope_hadamard_fp4_kernel<kFmt, kBN, kNoLoads, kFuse>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, K2Layout<kBN>::kSmemBytes);
}

// The fused-quantizer instance: clusters of two, launched cooperatively so
// that all CTAs are resident together (each waits for token rows that CTAs
// all over the grid quantize), and without programmatic serialization (it
// reads its inputs before any dependency wait).
template <int kFmt>
cudaError_t launch_fused(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const CUtensorMap& tm_q,
                         const GemmArgs& args, int pairs, cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pairs * kPair, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = K2Layout<256>::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_rope_hadamard_fp4_kernel<kFmt, 256, false, true>, tm_x, tm_w, tm_q, args);
}

template <int kFmt, int kBN, bool kNoLoads = false>
cudaError_t launch_one(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const CUtensorMap& tm_q,
                       const GemmArgs& args, int pairs, cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pair_config(pairs, K2Layout<kBN>::kSmemBytes, attr, stream);
  return cudaLaunchKernelEx(&cfg, gemm_rope_hadamard_fp4_kernel<kFmt, kBN, kNoLoads>, tm_x, tm_w, tm_q, args);
}

// Pairs to launch: at most max_pairs, and no more than the tiles need once
// each pair takes ceil(tiles / pairs) of them.
int launch_pairs(int tiles, int max_pairs) {
  const int p = tiles < max_pairs ? tiles : max_pairs;
  const int per = (tiles + p - 1) / p;
  return (tiles + per - 1) / per;
}

}  // namespace

int gemm_pair_size() { return kPair; }

cudaError_t gemm_setup_device(int* max_pairs) {
  for (cudaError_t err : {set_smem_attr<kFp4Mx, 256>(), set_smem_attr<kFp4MxOcp, 256>(), set_smem_attr<kFp4Nv, 256>(),
                          set_smem_attr<kFp4Mx, 128>(), set_smem_attr<kFp4MxOcp, 128>(), set_smem_attr<kFp4Nv, 128>(),
                          set_smem_attr<kFp4Mx, 256, true>(), set_smem_attr<kFp4Mx, 256, false, true>(),
                          set_smem_attr<kFp4MxOcp, 256, false, true>(), set_smem_attr<kFp4Nv, 256, false, true>()}) {
    if (err != cudaSuccess) return err;
  }
  // One CTA per SM for either width (tensor memory and registers), so the
  // wide instance's occupancy holds for both.
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pair_config(1, K2Layout<256>::kSmemBytes, attr, nullptr);
  return cudaOccupancyMaxActiveClusters(max_pairs, gemm_rope_hadamard_fp4_kernel<kFp4Mx, 256>, &cfg);
}

cudaError_t launch_gemm_rope_hadamard_fp4(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const CUtensorMap& tm_q,
                                          const GemmArgs& args, int tile_n, int fp4_format, int max_pairs,
                                          cudaStream_t stream) {
  const int pairs = launch_pairs(args.num_pair_tiles, max_pairs);
  if (tile_n == 128) {
    switch (fp4_format) {
      case kFp4Mx: return launch_one<kFp4Mx, 128>(tm_x, tm_w, tm_q, args, pairs, stream);
      case kFp4MxOcp: return launch_one<kFp4MxOcp, 128>(tm_x, tm_w, tm_q, args, pairs, stream);
      case kFp4Nv: return launch_one<kFp4Nv, 128>(tm_x, tm_w, tm_q, args, pairs, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (tile_n != 256) return cudaErrorInvalidValue;
  switch (fp4_format) {
    case kFp4Mx: return launch_one<kFp4Mx, 256>(tm_x, tm_w, tm_q, args, pairs, stream);
    case kFp4MxOcp: return launch_one<kFp4MxOcp, 256>(tm_x, tm_w, tm_q, args, pairs, stream);
    case kFp4Nv: return launch_one<kFp4Nv, 256>(tm_x, tm_w, tm_q, args, pairs, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_fused_quant(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const CUtensorMap& tm_q,
                                    const GemmArgs& args, int fp4_format, int max_pairs, cudaStream_t stream) {
  if (args.order != kOrderInterleaved || args.latent == nullptr || args.x_fp8 == nullptr ||
      args.x_sf_out == nullptr || args.ready == nullptr) {
    return cudaErrorInvalidValue;
  }
  const int pairs = launch_pairs(args.num_pair_tiles, max_pairs);
  if (pairs * kPair > kMaxFusedCtas) return cudaErrorInvalidValue;
  switch (fp4_format) {
    case kFp4Mx: return launch_fused<kFp4Mx>(tm_x, tm_w, tm_q, args, pairs, stream);
    case kFp4MxOcp: return launch_fused<kFp4MxOcp>(tm_x, tm_w, tm_q, args, pairs, stream);
    case kFp4Nv: return launch_fused<kFp4Nv>(tm_x, tm_w, tm_q, args, pairs, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_wait_selftest(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const CUtensorMap& tm_q,
                                      const GemmArgs& args, int max_pairs, cudaStream_t stream) {
  return launch_one<kFp4Mx, 256, true>(tm_x, tm_w, tm_q, args, launch_pairs(args.num_pair_tiles, max_pairs), stream);
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
