// K3: the fused indexer-Q projection for few tokens (M <= 128), with the MMA
// operands swapped: the weights are the MMA's M side and the tokens its N side.
//
// The TensorRT-LLM PR "Fuse DeepSeek-V4 Indexer Q projection with CuTe DSL"
// routes small token counts to a swapped-A/B kernel (dispatch thresholds:
// the swapped kernel wins through M = 8 on its hardware; description: a
// small-M variant next to the persistent kernel).  What it computes is the
// same as the large-M kernel: block-scaled FP8 GEMM, then per (token, head)
// RoPE -> Hadamard-128 -> FP4 E2M1 with 1x32 UE8M0 scales.
//
// Why a second kernel.  With few tokens the work is reading W (12.6 MB) and
// the fixed costs of a tile; the large-M kernel would still issue 256 x 256
// MMAs and run its epilogue on a whole 256-row tile.  Here:
//   * one cluster of two CTAs per head (128 CTAs).  Each CTA multiplies the
//     head's 128 rows of W (the MMA's A side, M = 128) by the token rows (the
//     B side: N = M rounded up to 16) over one half of K (6 of the 12
//     K-blocks) with the 1-SM MMA (tcgen05 kind::mxf8f6f4 block_scale); the
//     accumulators are FP32 in tensor memory.  Two instances: 64 token
//     columns for M <= 64 and 128 for 65 <= M <= 128, whose split-K exchange
//     buffer takes the place of the first two W and token stages (K3Layout);
//   * several MMA issuers: with one issuing thread the 24 MMAs of a CTA (32
//     cycles of tensor work each at N = 64) measured 100-160 cycles apart;
//     with the K-blocks dealt to three threads, each accumulating into its
//     own TMEM columns, the whole MMA phase took a third of the time.  The
//     epilogue adds the three partial sums;
//   * the token tile of a K-block is loaded as exactly M rows: rows M..N-1 of
//     the B side keep whatever shared memory held, which reaches only
//     accumulator columns M..N-1 (column n depends on B row n alone), and
//     those columns are never read.  (A box reaching past M would make TMA
//     fill the missing rows, measured to delay the load by ~0.7 us at M = 1);
//   * each CTA's share of W (96 KB) is loaded before the kernel waits for the
//     preceding grid (the quantizer, launched just before with programmatic
//     stream serialization): W does not depend on it, so its read overlaps
//     the quantizer;
//   * split-K exchange through distributed shared memory: token t is finished
//     by the CTA of K half t % 2, which keeps its own half's partial sums and
//     receives the other half's as asynchronous stores (st.async) counted on
//     one of its mbarriers;
//   * per token one warp runs the epilogue for the head: lane l holds dims
//     4l..4l+3, RoPE pairs (i, i+32) meet through one shuffle, the two
//     lowest Hadamard stages run in registers and the five others across
//     lanes with shuffles, each FP4 block of 32 dims is 8 lanes, and every
//     lane writes its 2 code bytes, so a warp stores the head's 64 code bytes
//     of the token at once.  A warp takes its tokens two at a time, so their
//     shuffle and sincos latencies overlap.
//
// Scale factors, as in the large-M kernel: the MMA applies one UE8M0 scale
// per 32 K per row; the instruction descriptor's scale-ID field (kb % 4)
// picks the byte of the packed word that holds K-block kb.  SFA carries the
// head's weight-block scale (the same for its 128 rows), SFB the scales of the
// token rows.
//
// Every mbarrier wait is bounded (GemmArgs::timeout_ns); a wait that gives up
// records its kind in this kernel's device status word.  No thread leaves a
// loop or the kernel early, so every thread of both CTAs reaches both uses of
// the cluster barrier exactly once: arrive after set-up (128 columns: once
// this CTA's MMAs on the exchange buffer's stages have completed), wait before
// the exchange (the peer is running); arrive after the exchange, wait at the
// end (the peer has issued its stores into this CTA, even when a wait gave
// up).

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "iq_fp4.cuh"
#include "iq_internal.h"
#include "iq_ptx.cuh"

namespace iq {

__device__ uint32_t g_iq_status_small_m;

namespace {

constexpr int kSplit = 2;                           // K halves: the CTAs of a cluster
constexpr int kKbPerCta = kNumKBlocks / kSplit;     // 6
constexpr int kWBytes = kHeadDim * 128;             // one head x one K-block: 16 KB
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
// MMA issuers (see above): issuer q takes K-blocks q, q + kIssuers, ... into
// accumulator q.
constexpr int kIssuers = 3;
constexpr int kKbPerIssuer = kKbPerCta / kIssuers;
constexpr uint32_t kAccCol = 0;                     // kIssuers x kN columns
constexpr int kNumBars = 2 * kKbPerCta + 5;
static_assert(kKbPerCta % kIssuers == 0 && kIssuers <= 6, "issuers");

// Token columns kN of the MMA: 64 (M <= 64) or 128 (65 <= M <= 128).
template <int kN>
struct K3Layout {
  static constexpr int kXBytes = kN * 128;                 // kN tokens x one K-block: 8 or 16 KB
  static constexpr int kSlots = kN / kSplit;               // tokens finished per CTA
  static constexpr int kTokPerWarp = kSlots / kWarps;      // tokens a warp finishes in step (3)
  static constexpr int kCols = kN / (kWarps / 4);          // token columns a warp drains in steps (1) and (2)
  static constexpr uint32_t kSfaCol = kIssuers * kN;       // + 8 g, 4 columns each
  static constexpr uint32_t kSfbCol = kSfaCol + 32;        // + 8 g, 4 columns each
  static constexpr uint32_t kTmemCols = kSfbCol + 32 <= 128 ? 128 : (kSfbCol + 32 <= 256 ? 256 : 512);
  // The split-K exchange buffer: per K half h, float [kSlots][128 dims] (the
  // partial sums of this CTA's tokens from half h).  With 128 token columns,
  // W (96 KB), the tokens (96 KB) and a separate 64 KB buffer do not fit, so
  // half 0 takes the place of the first kRedStages W stages and half 1 that of
  // the first kRedStages token stages: the MMAs of those K-blocks are issued
  // first, and each CTA arrives on the cluster barrier once its own have
  // completed, so neither CTA stores into the other before both are done
  // with those stages.
  static constexpr bool kRedInStages = kN > 64;
  static constexpr int kRedStages = 2;
  static constexpr int kRedHalfBytes = kSlots * kHeadDim * 4;
  // Shared-memory map (offsets from a 1024-byte aligned base).
  static constexpr int kOffW = 0;
  static constexpr int kOffX = kOffW + kKbPerCta * kWBytes;
  static constexpr int kOffSfa = kOffX + kKbPerCta * kXBytes;
  static constexpr int kOffSfb = kOffSfa + kScaleGroups * 128 * 4;
  static constexpr int kOffRed0 = kRedInStages ? kOffW : kOffSfb + kScaleGroups * 128 * 4;
  static constexpr int kOffRed1 = kRedInStages ? kOffX : kOffRed0 + kRedHalfBytes;
  static constexpr int kOffBar = kRedInStages ? kOffSfb + kScaleGroups * 128 * 4 : kOffRed1 + kRedHalfBytes;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack

  static_assert(kN == 64 || kN == 128, "token columns");
  static_assert(kSfbCol + 32 <= 512, "tensor memory");
  static_assert(kOffX % 1024 == 0 && kXBytes % 1024 == 0, "swizzled operand tiles need 1024-byte alignment");
  static_assert(kOffSfa % 16 == 0 && kOffSfb % 16 == 0 && kOffRed0 % 16 == 0 && kOffRed1 % 16 == 0 &&
                    kOffBar % 8 == 0,
                "alignment");
  // The stages that hold the buffer are K-blocks 0 .. kRedStages - 1, the
  // first K-block of issuers 0 .. kRedStages - 1.
  static_assert(!kRedInStages || (kRedHalfBytes <= kRedStages * kWBytes && kRedHalfBytes <= kRedStages * kXBytes &&
                                  kRedStages <= kIssuers),
                "exchange buffer inside the first stages");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kSlots % kWarps == 0 && kIssuers + 2 <= kWarps + 1, "warp roles");
  static_assert(kCols == 16 || kCols == 32, "16- or 32-column tensor-memory loads");
};

__device__ __forceinline__ void fail(volatile uint32_t* abort_flag, uint32_t bit) {
  atomicOr(&g_iq_status_small_m, bit);
  *abort_flag = 1u;
}

template <int kFmt, int kN>
__global__ void __launch_bounds__(kThreads, 1)
    small_m_rope_hadamard_fp4_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                                     const __grid_constant__ GemmArgs args) {
  using L = K3Layout<kN>;
  constexpr int kXBytes = L::kXBytes;
  constexpr int kTokPerWarp = L::kTokPerWarp;
  constexpr uint32_t kSfaCol = L::kSfaCol;
  constexpr uint32_t kSfbCol = L::kSfbCol;
  constexpr uint32_t kTmemCols = L::kTmemCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sW = smem + L::kOffW;
  uint8_t* sX = smem + L::kOffX;
  uint32_t* sSfa = reinterpret_cast<uint32_t*>(smem + L::kOffSfa);
  uint32_t* sSfb = reinterpret_cast<uint32_t*>(smem + L::kOffSfb);
  float* red0 = reinterpret_cast<float*>(smem + L::kOffRed0);   // K half 0's partial sums of this CTA's tokens
  float* red1 = reinterpret_cast<float*>(smem + L::kOffRed1);   // K half 1's
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* w_full = bars;                       // K-block i of W landed
  uint64_t* x_full = bars + kKbPerCta;           // K-block i of the tokens landed
  uint64_t* sf_full = bars + 2 * kKbPerCta;      // scale factors staged in shared memory
  uint64_t* sf_copied = sf_full + 1;             // scale factors copied into tensor memory
  uint64_t* mma_done = sf_full + 2;              // every issuer's MMAs completed
  uint64_t* red_full = sf_full + 3;              // both K halves' partial sums of this CTA's tokens landed
  uint64_t* first_done = sf_full + 4;            // the MMAs on the exchange buffer's stages completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kOffMisc + 4);

  // The next kernel of the stream may be scheduled now (it waits for this
  // one's completion before it touches memory).
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();       // the K half
  const int head = static_cast<int>(blockIdx.x) / kSplit;
  const int kb0 = static_cast<int>(rank) * kKbPerCta;
  const int M = args.M;
  const uint64_t timeout = args.timeout_ns;

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
    for (int i = 0; i < kKbPerCta; ++i) {
      mbar_init(&w_full[i], 1);
      mbar_init(&x_full[i], 1);
    }
    mbar_init(sf_full, 1);
    mbar_init(sf_copied, 1);
    mbar_init(mma_done, kIssuers);
    mbar_init(red_full, 1);
    mbar_init(first_done, L::kRedStages);
    *abort_flag = 0u;
    fence_mbar_init();
    // This CTA finishes the tokens t < M with t % 2 == rank; the peer's K
    // half of each arrives as 128 floats (this CTA's own half is stored
    // locally).
    const uint32_t own_tokens = static_cast<uint32_t>((M - static_cast<int>(rank) + 1) / 2);
    mbar_arrive_expect_tx(red_full, own_tokens * kHeadDim * 4u);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // This CTA is running: the peer may address its shared memory once it has
  // passed the matching wait (just before the split-K exchange).  With the
  // exchange buffer in the first stages the arrive comes once this CTA's
  // MMAs on them have completed.
  if constexpr (!L::kRedInStages) cluster_arrive_relaxed();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int i = 0; i < kKbPerCta; ++i) {
        mbar_arrive_expect_tx(&w_full[i], kWBytes);
        tma_load_2d(sW + i * kWBytes, &tm_w, &w_full[i], (kb0 + i) * 128, head * kHeadDim);
      }
      // The FP8 tokens are the preceding grid's output.
      grid_dependency_wait();
      for (int i = 0; i < kKbPerCta; ++i) {
        mbar_arrive_expect_tx(&x_full[i], static_cast<uint32_t>(M) * 128u);
        tma_load_2d(sX + i * kXBytes, &tm_x, &x_full[i], (kb0 + i) * 128, 0);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------ scale-factor staging
    // tcgen05.cp 32x128b layout: word [r * 4 + c] of a group holds row
    // c * 32 + r.  SFA: the head's weight scales (all 128 rows alike); SFB:
    // the activation scale words of tokens 0..63 (0 past M: those columns
    // hold zeros and are never stored).
#pragma unroll
    for (int g = 0; g < kScaleGroups; ++g) {
      const uint8_t* ws = args.w_sf + head * kNumKBlocks + 4 * g;
      const uint32_t w = static_cast<uint32_t>(__ldg(ws)) | (static_cast<uint32_t>(__ldg(ws + 1)) << 8) |
                         (static_cast<uint32_t>(__ldg(ws + 2)) << 16) | (static_cast<uint32_t>(__ldg(ws + 3)) << 24);
      *reinterpret_cast<uint4*>(sSfa + g * 128 + lane * 4) = make_uint4(w, w, w, w);
    }
    grid_dependency_wait();
#pragma unroll
    for (int g = 0; g < kScaleGroups; ++g) {
      uint32_t r[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int m = c * 32 + lane;
        r[c] = m < M ? ld_dependent_u32(args.x_sf + static_cast<long long>(g) * args.m_al + m) : 0u;
      }
      *reinterpret_cast<uint4*>(sSfb + g * 128 + lane * 4) = make_uint4(r[0], r[1], r[2], r[3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(sf_full);
  } else if (warp - (warp == 1 ? 1 : 2) < kIssuers) {
    // ------------------------------------------------------- MMA issuers
    // Issuer q is warp 1 (q = 0), then warps 3, 4, ...; issuer 0 first
    // copies the scale factors into tensor memory.
    const int q = warp == 1 ? 0 : warp - 2;
    if (lane == 0) {
      bool ok = true;
      bool first_sent = false;   // this issuer's arrival on first_done
      if (q == 0) {
        ok = mbar_wait(sf_full, 0, timeout);
        if (ok) {
          tc_fence_after_sync();
#pragma unroll
          for (int g = 0; g < kScaleGroups; ++g) {
            tc_cp_32x128b_warpx4(tmem + kSfaCol + 8 * g, smem_desc_sf(smem_u32(sSfa + g * 128)));
            tc_cp_32x128b_warpx4(tmem + kSfbCol + 8 * g, smem_desc_sf(smem_u32(sSfb + g * 128)));
          }
        }
        // Arrives once the copies completed (also when the wait gave up).
        tc_commit(sf_copied);
      }
      ok = ok && mbar_wait(sf_copied, 0, timeout);
      if (ok) {
        tc_fence_after_sync();
        const uint64_t adesc0 = smem_desc_sw128(smem_u32(sW));
        const uint64_t bdesc0 = smem_desc_sw128(smem_u32(sX));
        // The MMA's N: the token count rounded up to 16 (the step of N at
        // M = 128); accumulator columns past it are not written, and the
        // epilogue reads only columns below M.
        const int n_cols = min(kN, max(16, (M + 15) & ~15));
        const uint32_t idesc0 = idesc_mxf8_e4m3(kHeadDim, n_cols, 0, 0);
        const uint32_t acc = tmem + kAccCol + static_cast<uint32_t>(q * kN);
        for (int n = 0; n < kKbPerIssuer; ++n) {
          const int i = q + n * kIssuers;
          // This issuer's first K-block is done with: its completion frees the
          // exchange buffer's stages (see K3Layout).
          if (L::kRedInStages && n == 1 && q < L::kRedStages) {
            tc_commit(first_done);
            first_sent = true;
          }
          if (!mbar_wait(&w_full[i], 0, timeout) || !mbar_wait(&x_full[i], 0, timeout)) {
            ok = false;
            break;
          }
          const int kb = kb0 + i;
          const uint32_t sfid = static_cast<uint32_t>(kb & 3);
          const uint32_t idesc = idesc0 | (sfid << 4) | (sfid << 29);
          const uint32_t sf_off = 8u * static_cast<uint32_t>(kb >> 2);
          const uint64_t adesc = adesc0 + static_cast<uint64_t>(i * (kWBytes >> 4));
          const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(i * (kXBytes >> 4));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // advance 32 bytes along K inside the 128-byte swizzle atom
            tc_mma_mxf8(acc, adesc + 2 * k, bdesc + 2 * k, idesc, tmem + kSfaCol + sf_off, tmem + kSfbCol + sf_off,
                        (n | k) != 0);
          }
        }
      }
      if (!ok) fail(abort_flag, kStatusMmaWait);
      // A wait that gave up may have left first_done without this issuer's
      // arrival; add it (it arrives once whatever was issued has completed).
      if (L::kRedInStages && q < L::kRedStages && !first_sent) tc_commit(first_done);
      // Arrives once everything this thread issued has completed (also when
      // a wait gave up before any MMA was issued).
      tc_commit(mma_done);
    }
    __syncwarp();
  }

  // -------------------------------------------------------------- epilogue
  // Per-token inputs of step (3), loaded while the MMAs run: this warp's
  // tokens t = 2 (warp + 8 j) + K half, their positions (lanes 0..15 rotate),
  // and the RoPE frequencies of dims 4 (l % 8) + k in turns per position unit
  // (lanes 0..7 hold the first element of each NeoX pair, 8..15 the second).
  // Positions are read after the wait like every other input (besides W and
  // its scales); the epilogue warps are idle until the MMAs complete anyway.
  grid_dependency_wait();
  int tok_index[kTokPerWarp];
  bool tok_valid[kTokPerWarp];
  float tok_pos[kTokPerWarp];
#pragma unroll
  for (int j = 0; j < kTokPerWarp; ++j) {
    tok_index[j] = 2 * (warp + j * kWarps) + static_cast<int>(rank);
    tok_valid[j] = tok_index[j] < M;
    tok_pos[j] =
        (tok_valid[j] && lane < 16) ? static_cast<float>(static_cast<int>(ld_dependent_u32(args.pos + tok_index[j]))) : 0.f;
  }
  // The RoPE rotation of each token's dims (lanes 0..15), computed while the
  // MMAs run: cos and (sign-adjusted) sin of angle = position * frequency.
  // The angle is reduced in turns with a two-float product of position and
  // frequency (the rounding to an integer uses the 1.5 * 2^23 shift, exact
  // for |turns| < 2^22), then scaled to radians in [-pi, pi].
  const float rope_sign = lane < 8 ? -1.f : 1.f;
  float rcos[kTokPerWarp][4], rsin[kTokPerWarp][4];
  {
    float fhi[4], flo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      fhi[k] = args.rope.hi[4 * (lane & 7) + k];
      flo[k] = args.rope.lo[4 * (lane & 7) + k];
    }
#pragma unroll
    for (int j = 0; j < kTokPerWarp; ++j) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float th = __fmul_rn(tok_pos[j], fhi[k]);
        float tl = __fmaf_rn(tok_pos[j], fhi[k], -th);
        tl = __fmaf_rn(tok_pos[j], flo[k], tl);
        const float rn = __fsub_rn(__fadd_rn(th, 12582912.0f), 12582912.0f);
        const float ang = __fmul_rn(__fadd_rn(__fsub_rn(th, rn), tl), kTwoPi);
        float sn, cs;
        __sincosf(ang, &sn, &cs);
        rcos[j][k] = cs;
        rsin[j][k] = rope_sign * sn;
      }
    }
  }

  // (1) This CTA's partial sums over its K half: TMEM lane d = dim d of the
  // head, column j of accumulator q = token j.
  if constexpr (L::kRedInStages) {
    // This CTA's MMAs no longer read the exchange buffer's stages: the peer
    // may store into them once it has passed the matching wait.  The arrive
    // publishes no data, only that the wait above has returned, so it is
    // relaxed (a release arrive here measured ~0.75 us).
    if (!mbar_wait(first_done, 0, timeout)) fail(abort_flag, kStatusEpilogueWait);
    __syncwarp();
    cluster_arrive_relaxed();
  }
  const bool got = mbar_wait(mma_done, 0, timeout);
  if (!got) fail(abort_flag, kStatusEpilogueWait);
  __syncwarp();   // the lanes left the polling loop separately; tcgen05.ld is .sync.aligned
  tc_fence_after_sync();
  // Warp w drains TMEM lanes 32 (w % 4).. and the 16-column chunks
  // w / 4, w / 4 + 4, ... (token columns 16 c .. 16 c + 15 of chunk c), so
  // that with fewer tokens than columns every warp still takes a share.
  const int quad = warp & 3;
  constexpr int kCols = L::kCols;
  constexpr int kChunks = kCols / 16;
  const int chunk0 = warp >> 2;
  const int d = quad * 32 + lane;
  float v[kCols];
  {
    const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + kAccCol;
    // Per chunk that holds a token: the three accumulators' loads issued
    // together, then one wait.
    static_assert(kIssuers == 3, "three accumulators per chunk");
#pragma unroll
    for (int k = 0; k < kChunks; ++k) {
      const int c0 = 16 * (chunk0 + 4 * k);
      if (c0 >= M) break;   // warp-uniform; chunks fill in order
      float w[48];
#pragma unroll
      for (int q = 0; q < kIssuers; ++q) tmem_ld_32x32b_x16(taddr + static_cast<uint32_t>(q * kN + c0), w + 16 * q);
      tmem_ld_wait(w);
      tmem_ld_wait16(w + 32);
#pragma unroll
      for (int j = 0; j < 16; ++j) v[16 * k + j] = w[j] + w[16 + j] + w[32 + j];
    }
  }
  tc_fence_before_sync();

  // (2) Split-K exchange.  Token t is finished in slot t / 2 by CTA t % 2;
  // this CTA's partial goes to that CTA's buffer of K half `rank`: for its
  // own tokens by plain shared-memory stores (visible after the block
  // barrier below), for the peer's as asynchronous stores counted on the
  // peer's red_full barrier (no cluster-scope release fence, which costs ~1K
  // cycles here).
  cluster_wait();   // the peer is running (its barriers are initialized; with
                    // the buffer in the first stages, its MMAs on them
                    // have completed)
  float* red_own = rank == 0 ? red0 : red1;
  const uint32_t peer = rank ^ 1u;
  const uint32_t red_peer = mapa_shared(smem_u32(red_own) + static_cast<uint32_t>(d * 4), peer);
  const uint32_t bar_peer = mapa_shared(smem_u32(red_full), peer);
#pragma unroll
  for (int k = 0; k < kChunks; ++k) {
    const int c0 = 16 * (chunk0 + 4 * k);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int t = c0 + j;   // c0 is even: t % 2 == j % 2
      if (t < M) {
        if (static_cast<uint32_t>(j & 1) == rank)
          red_own[(t >> 1) * kHeadDim + d] = v[16 * k + j];
        else
          st_async_cluster_f32(red_peer + static_cast<uint32_t>((t >> 1) * kHeadDim * 4), v[16 * k + j], bar_peer);
      }
    }
  }
  const bool red_ok = mbar_wait(red_full, 0, timeout);
  if (!red_ok) fail(abort_flag, kStatusEpilogueWait);
  // Second use of the cluster barrier: this CTA has issued every store into
  // the peer.  Its wait, at the very end, keeps each CTA resident until the
  // peer has issued all of its stores into it (see the end of the kernel).
  cluster_arrive_relaxed();
  // Every thread has read its tensor memory: release it.
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }

  // (3) Per token one warp: lane l holds dims 4l..4l+3 of the head.  A warp
  // takes its tokens (slots warp, warp + kWarps, ...) two at a time, so the
  // shuffle and sincos latencies of one token overlap those of the other.
  // Slots fill in order, so a pair whose first slot holds no token ends the
  // warp's work.
  constexpr int kLanesPerBlock = Fp4Layout<kFmt>::kBlock / 4;
  static_assert(kTokPerWarp % 2 == 0, "token pairs");
#pragma unroll
  for (int g = 0; g < kTokPerWarp; g += 2) {
    if (!tok_valid[g]) break;   // warp-uniform
    float x[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int u = warp + (g + j) * kWarps;
      const float4 a = reinterpret_cast<const float4*>(red0 + u * kHeadDim)[lane];
      const float4 b = reinterpret_cast<const float4*>(red1 + u * kHeadDim)[lane];
      x[j][0] = a.x + b.x;
      x[j][1] = a.y + b.y;
      x[j][2] = a.z + b.z;
      x[j][3] = a.w + b.w;
    }
    // NeoX RoPE on dims 0..63 (lanes 0..15): x1' = x1 c - x2 s, x2' = x2 c + x1 s.
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float y[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) y[k] = __shfl_xor_sync(0xFFFFFFFFu, x[j][k], 8);
      if (lane < 16) {
#pragma unroll
        for (int k = 0; k < 4; ++k) x[j][k] = __fmaf_rn(x[j][k], rcos[g + j][k], __fmul_rn(y[k], rsin[g + j][k]));
      }
    }
    // Fast Walsh-Hadamard transform in Sylvester order (unscaled): dim bits 0
    // and 1 inside the lane, bits 2..6 across lanes (partner lane l ^ m; the
    // lane with the bit clear keeps a + b, the other a - b).
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float h0 = x[j][0] + x[j][1], h1 = x[j][0] - x[j][1];
      const float h2 = x[j][2] + x[j][3], h3 = x[j][2] - x[j][3];
      x[j][0] = h0 + h2;
      x[j][1] = h1 + h3;
      x[j][2] = h0 - h2;
      x[j][3] = h1 - h3;
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const float sg = (lane & m) ? -1.f : 1.f;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float p = __shfl_xor_sync(0xFFFFFFFFu, x[j][k], m);
          x[j][k] = __fmaf_rn(sg, x[j][k], p);
        }
      }
    }
    // FP4 of z = v / sqrt(128): a block of 32 dims is lanes 8b..8b+7 (MX
    // variants), a block of 16 dims lanes 4b..4b+3 (NVFP4-style).
    float amax[2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
      amax[j] = fmaxf(fmaxf(fabsf(x[j][0]), fabsf(x[j][1])), fmaxf(fabsf(x[j][2]), fabsf(x[j][3])));
#pragma unroll
    for (int m = 1; m < kLanesPerBlock; m <<= 1) {
#pragma unroll
      for (int j = 0; j < 2; ++j) amax[j] = fmaxf(amax[j], __shfl_xor_sync(0xFFFFFFFFu, amax[j], m));
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (!tok_valid[g + j]) continue;   // warp-uniform
      const long long t = tok_index[g + j];
      uint32_t codes, sbyte;
      if constexpr (kFmt != kFp4Nv) {
        const int e = fp4_block_exponent<kFmt>(amax[j] * kInvSqrt128);
        const float kq = fp4_code_factor(e);
        codes = cvt_e2m1x4(x[j][0] * kq, x[j][1] * kq, x[j][2] * kq, x[j][3] * kq);
        sbyte = static_cast<uint32_t>(e + 127);
      } else {
        sbyte = nvfp4_code(fmaxf(amax[j] * kInvSqrt128, kAmaxFloor) * kSixth);
        const float kq = e4m3_reciprocal(sbyte) * kInvSqrt128;
        codes = cvt_e2m1x4(x[j][0] * kq, x[j][1] * kq, x[j][2] * kq, x[j][3] * kq);
      }
      // Byte 64 h + 2 l + i of the token's row holds dims 4l + 2i, 4l + 2i + 1.
      reinterpret_cast<uint16_t*>(args.q_fp4 + t * (kQDim / 2) + head * 64)[lane] = static_cast<uint16_t>(codes);
      if (lane % kLanesPerBlock == 0)
        args.q_sf[t * Fp4Layout<kFmt>::kScaleBytesPerToken + head * Fp4Layout<kFmt>::kBlocksPerHead +
                  lane / kLanesPerBlock] = static_cast<uint8_t>(sbyte);
      if (args.q_pre != nullptr) {
        reinterpret_cast<float4*>(args.q_pre + t * kQDim + head * kHeadDim)[lane] =
            make_float4(x[j][0] * kInvSqrt128, x[j][1] * kInvSqrt128, x[j][2] * kInvSqrt128, x[j][3] * kInvSqrt128);
      }
    }
  }

  // Every load landed before the MMAs that read it completed, and the peer's
  // stores into this CTA's shared memory completed before red_full did; this
  // CTA's stores into the peer completed before the peer passed its red_full
  // wait, so neither CTA touches the other's shared memory after the exchange.
  // If a red_full wait gave up, the peer may be late: the cluster wait below
  // returns once the peer has issued all its stores into this CTA (its arrive
  // follows them), and a bounded second wait on red_full lets them land before
  // this CTA's shared memory is released.
  cluster_wait();
  if (!red_ok && threadIdx.x == 0) {
    if (!mbar_wait(red_full, 0, timeout)) fail(abort_flag, kStatusTeardownWait);
  }
  __syncthreads();
}

cudaLaunchConfig_t small_m_config(cudaLaunchAttribute* attr, int smem_bytes, cudaStream_t stream) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kSplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kNumHeads * kSplit, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

template <int kN>
cudaError_t small_m_setup_width() {
  for (const void* fn : {reinterpret_cast<const void*>(small_m_rope_hadamard_fp4_kernel<kFp4Mx, kN>),
                         reinterpret_cast<const void*>(small_m_rope_hadamard_fp4_kernel<kFp4MxOcp, kN>),
                         reinterpret_cast<const void*>(small_m_rope_hadamard_fp4_kernel<kFp4Nv, kN>)}) {
    const cudaError_t err =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, K3Layout<kN>::kSmemBytes);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

template <int kN>
cudaError_t launch_width(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const GemmArgs& args, int fp4_format,
                         cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = small_m_config(attr, K3Layout<kN>::kSmemBytes, stream);
  switch (fp4_format) {
    case kFp4Mx: return cudaLaunchKernelEx(&cfg, small_m_rope_hadamard_fp4_kernel<kFp4Mx, kN>, tm_x, tm_w, args);
    case kFp4MxOcp:
      return cudaLaunchKernelEx(&cfg, small_m_rope_hadamard_fp4_kernel<kFp4MxOcp, kN>, tm_x, tm_w, args);
    case kFp4Nv: return cudaLaunchKernelEx(&cfg, small_m_rope_hadamard_fp4_kernel<kFp4Nv, kN>, tm_x, tm_w, args);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t small_m_setup_device() {
  const cudaError_t err = small_m_setup_width<64>();
  return err != cudaSuccess ? err : small_m_setup_width<128>();
}

cudaError_t launch_small_m_rope_hadamard_fp4(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const GemmArgs& args,
                                             int fp4_format, cudaStream_t stream) {
  if (args.M < 1 || args.M > kSmallMMax) return cudaErrorInvalidValue;
  return args.M <= 64 ? launch_width<64>(tm_x, tm_w, args, fp4_format, stream)
                      : launch_width<128>(tm_x, tm_w, args, fp4_format, stream);
}

cudaError_t read_small_m_status(uint32_t* flags, bool reset) {
  uint32_t v = 0;
  cudaError_t err = cudaMemcpyFromSymbol(&v, g_iq_status_small_m, sizeof(v));
  if (err != cudaSuccess) return err;
  if (flags) *flags = v;
  if (reset) {
    const uint32_t zero = 0;
    err = cudaMemcpyToSymbol(g_iq_status_small_m, &zero, sizeof(zero));
  }
  return err;
}

}  // namespace iq
