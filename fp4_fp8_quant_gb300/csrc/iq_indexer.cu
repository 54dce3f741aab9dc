// The consumer of the prepared Q: the sparse-attention indexer's scores and
// its top-k selection (TokenSpeed PR "perf(deepseek-v4): accelerate indexer Q
// and packed FP8 quantization", Summary and Prefill host-sync cleanup: the
// indexer top-k written straight to its destination).  The pages name this
// consumer without its formulas or layouts; the kernels follow these readings:
//   score  I[t, s] = sum_h w[t, h] * max(0, q(t, h) . k(s)) over the 64 heads,
//          q(t, h) head h of token t's FP4 Q as iq_prepare_q writes it, k(s)
//          the 128-dim key of cached token s in the same MXFP4 format (E2M1
//          codes [N, 64] bytes, UE8M0 scale bytes [N, 4]); keys s < L[t] are
//          visible to query t;
//   top-k  the k visible keys with the largest scores, ties to the smaller
//          key index, as int32 indices in ascending order, -1 padded.
//
// K5 indexer_logits_kernel.  A dense FP4 contraction, so on the tensor cores:
// tcgen05.mma kind::mxf4 block_scale (E2M1 x E2M1, UE8M0 per 32 K) with the
// keys on the MMA's M side (128 per tile) and two query tokens x 64 heads on
// its N side (128), K = 128 in two MMAs of 64.  Each FP32 accumulator lane is
// one key and holds all 64 heads of both tokens, so the ReLU and the weighted
// sum over the heads stay inside one thread of the epilogue.  Warp roles (352
// threads): warps 0 and 10 decide the tile sequence and fill alternate
// stages of a 6-stage ring -- key and query tiles by TMA (64-byte rows,
// 64-byte swizzle), their scale words and the pair's weights by asynchronous
// copies, the tile's metadata, two end markers after the last tile; warp 1
// owns tensor memory and issues the scale copies and MMAs of every tile, in
// order, into three accumulator buffers; warps 2..9, two groups of four (one
// warp per 32-lane quarter of tensor memory) taking alternate tiles, drain an
// accumulator and form 32 keys' scores for both tokens from the stage's
// weights.
// Tiles (key block, token pair) are dealt to the CTAs in chunks of 8
// consecutive token pairs of one key block, chunk c to CTA c mod grid; the
// producer skips the pairs that can see no key of the block.
//
// K6 indexer_topk_kernel.  One CTA per query row: radix selection of the k-th
// largest score over order-preserving 32-bit keys (11, 11, then 10 bits,
// histograms in shared memory; a row of up to 12288 keys is read once and
// kept in shared memory), then a pass in index order over contiguous
// per-thread segments that writes the keys above the threshold and the first
// (smallest-index) keys equal to it.
//
// Every mbarrier wait is bounded (timeout_ns); a wait that gives up records
// its kind in this file's status word and raises a CTA abort flag.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "iq_internal.h"
#include "iq_ptx.cuh"

namespace iq {

__device__ uint32_t g_iq_status_indexer;

namespace {

constexpr int kKeysPerTile = 128;                    // MMA M
constexpr int kTokensPerTile = 2;
constexpr int kRowsB = kTokensPerTile * kNumHeads;   // MMA N = 128
constexpr int kRowBytes = kHeadDim / 2;              // 64: one packed FP4 head / key
constexpr int kTileBytes = kKeysPerTile * kRowBytes; // 8 KB, A and B alike
constexpr int kStages = 6;
constexpr int kAccBufs = 3;
constexpr int kChunkPairs = 8;                       // token pairs per chunk of tiles
constexpr int kEpiWarps = 8;                         // two groups of four, alternate tiles
constexpr int kGroupWarps = 4;
constexpr int kProducerWarp2 = 2 + kEpiWarps;        // the second producer (odd tiles)
constexpr int kThreads = (3 + kEpiWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfaCol = kAccBufs * kRowsB;      // 384 + 8 b
constexpr uint32_t kSfbCol = kSfaCol + 32;           // 416 + 8 b
static_assert(kSfbCol + 8 * kAccBufs <= kTmemCols, "tensor memory columns");

// Shared memory per stage: A tile (keys), B tile (the pair's query heads),
// their scale words in the tcgen05.cp 32x128b layout (512 B each), the pair's
// weights (2 x 64 floats) and the tile's metadata.  The producer decides the
// tile sequence and writes each tile's metadata into its stage; the MMA
// issuer and the epilogue follow the stages, so only the producer reads the
// visible lengths.  A stage is released by the MMAs and the four warps of
// the epilogue group that takes the tile (they read its weights and metadata).
constexpr int kOffSfa = 2 * kTileBytes;
constexpr int kOffSfb = kOffSfa + 512;
constexpr int kOffW = kOffSfb + 512;
constexpr int kOffMeta = kOffW + kTokensPerTile * kNumHeads * 4;
constexpr int kStageBytes = 18 * 1024;
static_assert(kOffMeta + 16 <= kStageBytes && kStageBytes % 1024 == 0, "stage layout");
constexpr int kOffBar = kStages * kStageBytes;
constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
// Two producer warps fill alternate tiles (stage s belongs to producer s % 2).
// Each completes one of its stages (its last arrive) this many of its own
// tiles after issuing the stage's asynchronous copies, so their latency
// overlaps later tiles.
constexpr int kProducers = 2;
constexpr int kCopyLag = 2;
static_assert(kStages % kProducers == 0 && kCopyLag < kStages / kProducers, "a stage's arrive precedes its reuse");

struct IndexerArgs {
  const uint32_t* k_sf;   // [N] scale words (4 UE8M0 bytes per key)
  const uint32_t* q_sf;   // [M * 64] scale words (4 per (token, head))
  const float* w;         // [M][64]
  const int32_t* len;     // [M]
  float* logits;          // [M][ld]
  long long ld;
  int M, N;
  int key_blocks, pairs, chunks_per_block, num_chunks;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ void fail(volatile uint32_t* abort_flag, uint32_t bit) {
  atomicOr(&g_iq_status_indexer, bit);
  *abort_flag = 1u;
}

// Lengths of the 16 tokens of a chunk's 8 pairs, one per lane (lanes 0..15),
// clamped to [0, N]; 0 past M.
__device__ __forceinline__ int chunk_lengths(const IndexerArgs& a, int ch, int lane) {
  if (ch >= a.num_chunks || lane >= 2 * kChunkPairs) return 0;
  const int kb = ch / a.chunks_per_block;
  const int t = (ch - kb * a.chunks_per_block) * 2 * kChunkPairs + lane;
  if (t >= a.M) return 0;
  const int L = __ldg(a.len + t);
  return L < 0 ? 0 : (L > a.N ? a.N : L);
}

__global__ void __launch_bounds__(kThreads, 1)
    indexer_logits_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ IndexerArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = bars;                          // stage s filled (TMA bytes + the producer's arrive)
  uint64_t* empty = bars + kStages;               // stage s consumed by the MMAs and the epilogue
  uint64_t* acc_full = bars + 2 * kStages;        // accumulator b complete
  uint64_t* acc_empty = acc_full + kAccBufs;      // accumulator b drained by the 8 epilogue warps
  uint64_t* final_bar = acc_empty + kAccBufs;     // every MMA issued by this CTA completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t timeout = args.timeout_ns;

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_q);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1 + kGroupWarps);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kGroupWarps);
    }
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
  // The queries' FP4 Q may be the preceding kernel's output.
  grid_dependency_wait();

  if (warp == 0 || warp == kProducerWarp2) {
    // ----------------------------------------------------------- producers
    // Tiles: chunks ch = blockIdx.x, + gridDim.x, ...; in each, the token
    // pairs g0 .. g0 + 7 against key block kb, skipping pairs that cannot
    // see any key of the block; then two end markers (g = -1).  Both
    // producers walk the whole sequence; producer p fills the tiles with
    // it % 2 == p.  A stage's asynchronous copies (scale words, weights) are
    // waited for kCopyLag of the producer's own tiles later; then the stage is
    // arrived.
    const int p = warp == 0 ? 0 : 1;
    uint32_t issued_mask = 0, issued_phase = 0;
    int it = 0, own = 0;
    bool ok = true;
    auto complete_stage = [&](int j) {   // global tile j's copies have landed
      uint8_t* st = smem + (j % kStages) * kStageBytes;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int g = reinterpret_cast<const volatile int*>(st + kOffMeta)[1];
        if (g >= 0) {
          mbar_arrive_expect_tx(&full[j % kStages], 2 * kTileBytes);
        } else {
          mbar_arrive(&full[j % kStages]);   // the end marker has no tile loads
        }
      }
    };
    // Global tile index of this producer's own tile n.
    auto own_tile = [&](int n) { return n * kProducers + p; };
    auto stage_tile = [&](int kb, int g, int L0, int L1) -> bool {
      const int mine = (it % kProducers) == p;
      const int s = it % kStages;
      const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
      ++it;
      if (!mine) return true;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&empty[s], ph ^ 1u, timeout))) {
        if (lane == 0) fail(abort_flag, kStatusProducerWait);
        return false;
      }
      uint8_t* st = smem + s * kStageBytes;
      if (g >= 0) {
        // Scale words straight into the tcgen05.cp 32x128b layout, word
        // [r * 4 + c] = row c * 32 + r (lane r copies rows r, 32 + r, ...);
        // rows past the data zero-filled.  The pair's weights, 16 bytes per lane.
        uint32_t* sfa = reinterpret_cast<uint32_t*>(st + kOffSfa);
        uint32_t* sfb = reinterpret_cast<uint32_t*>(st + kOffSfb);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int key = kb * kKeysPerTile + c * 32 + lane;
          cp_async_4(sfa + lane * 4 + c, args.k_sf + (key < args.N ? key : 0), key < args.N ? 4u : 0u);
          const long long qrow = static_cast<long long>(g) * kRowsB + c * 32 + lane;
          const bool qin = qrow < static_cast<long long>(args.M) * kNumHeads;
          cp_async_4(sfb + lane * 4 + c, args.q_sf + (qin ? qrow : 0), qin ? 4u : 0u);
        }
        const bool win = 2 * g + lane / 16 < args.M;
        cp_async_16(st + kOffW + lane * 16, args.w + (win ? static_cast<long long>(2 * g) * kNumHeads + lane * 4 : 0),
                    win ? 16u : 0u);
      }
      cp_async_commit();
      if (lane == 0) {
        *reinterpret_cast<int4*>(st + kOffMeta) = make_int4(kb, g, L0, L1);
        if (g >= 0) {
          tma_load_2d(st, &tm_k, &full[s], 0, kb * kKeysPerTile);
          tma_load_2d(st + kTileBytes, &tm_q, &full[s], 0, g * kRowsB);
          issued_mask |= 1u << s;
          issued_phase = (issued_phase & ~(1u << s)) | (ph << s);
        }
      }
      ++own;
      if (own > kCopyLag) {
        cp_async_wait<kCopyLag>();
        complete_stage(own_tile(own - 1 - kCopyLag));
      }
      return true;
    };
    int lv = chunk_lengths(args, blockIdx.x, lane);
    for (int ch = blockIdx.x; ch < args.num_chunks && ok; ch += gridDim.x) {
      const int lv_next = chunk_lengths(args, ch + gridDim.x, lane);   // in flight during this chunk
      const int kb = ch / args.chunks_per_block;
      const int gbase = (ch - kb * args.chunks_per_block) * kChunkPairs;
      for (int j = 0; j < kChunkPairs && ok; ++j) {
        const int g = gbase + j;
        const int L0 = __shfl_sync(0xFFFFFFFFu, lv, 2 * j);
        const int L1 = __shfl_sync(0xFFFFFFFFu, lv, 2 * j + 1);
        if (g >= args.pairs || kb * kKeysPerTile >= max(L0, L1)) continue;
        if (__any_sync(0xFFFFFFFFu, *abort_flag != 0u)) {
          ok = false;
          break;
        }
        ok = stage_tile(kb, g, L0, L1);
      }
      lv = lv_next;
    }
    // Two end markers (g = -1), one for each MMA issuer and epilogue group
    // (they take alternate tiles), then every own stage still waiting for its
    // copies.
    if (ok) ok = stage_tile(0, -1, 0, 0);
    if (ok) ok = stage_tile(0, -1, 0, 0);
    cp_async_wait<0>();
    for (int n = own - kCopyLag > 0 ? own - kCopyLag : 0; n < own; ++n) complete_stage(own_tile(n));
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if (((issued_mask >> s) & 1u) && !mbar_wait(&empty[s], (issued_phase >> s) & 1u, 2 * timeout))
          fail(abort_flag, kStatusTeardownWait);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One issuer takes every tile in order, so that each tile's MMAs depend
    // only on earlier tiles: with two issuers on alternate tiles sharing the
    // three accumulator buffers, the two halves of the pipeline could end up
    // waiting on each other.  It passes both end markers on, then stops.
    if (lane == 0) {
      const uint32_t idesc_k0 = idesc_mxf4_e2m1(kKeysPerTile, kRowsB, 0, 0);
      const uint32_t idesc_k1 = idesc_mxf4_e2m1(kKeysPerTile, kRowsB, 2, 2);
      int markers = 0;
      for (int it = 0;; ++it) {
        const int s = it % kStages;
        const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
        const int b = it % kAccBufs;
        const uint32_t aph = static_cast<uint32_t>(it / kAccBufs) & 1u;
        if (*abort_flag) break;
        if (!mbar_wait(&full[s], ph, timeout) || !mbar_wait(&acc_empty[b], aph ^ 1u, timeout)) {
          fail(abort_flag, kStatusMmaWait);
          break;
        }
        tc_fence_after_sync();
        uint8_t* st = smem + s * kStageBytes;
        const int g = reinterpret_cast<const volatile int*>(st + kOffMeta)[1];
        if (g >= 0) {
          const uint32_t sfa = tmem + kSfaCol + 8u * b;
          const uint32_t sfb = tmem + kSfbCol + 8u * b;
          tc_cp_32x128b_warpx4(sfa, smem_desc_sf(smem_u32(st + kOffSfa)));
          tc_cp_32x128b_warpx4(sfb, smem_desc_sf(smem_u32(st + kOffSfb)));
          const uint64_t adesc = smem_desc_sw64(smem_u32(st));
          const uint64_t bdesc = smem_desc_sw64(smem_u32(st + kTileBytes));
          const uint32_t d = tmem + static_cast<uint32_t>(b * kRowsB);
          // K = 128: dims 0..63 (scale bytes 0, 1), then dims 64..127 (bytes 2,
          // 3), 32 bytes further along each 64-byte row.
          tc_mma_mxf4(d, adesc, bdesc, idesc_k0, sfa, sfb, 0u);
          tc_mma_mxf4(d, adesc + 2, bdesc + 2, idesc_k1, sfa, sfb, 1u);
        }
        tc_commit(&empty[s]);
        tc_commit(&acc_full[b]);   // also passes an end marker on to the epilogue
        if (g < 0 && ++markers == 2) break;
      }
      tc_commit(final_bar);
      if (!mbar_wait(final_bar, 0, 2 * timeout)) fail(abort_flag, kStatusTeardownWait);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Group (warp - 2) / 4 takes the tiles of its parity; each warp drains
    // TMEM lanes 32 quad .. 32 quad + 31 (32 keys) for both tokens.
    const int quad = warp & 3;
    const int group = (warp - 2) >> 2;
    for (int it = group;; it += 2) {
      const int s = it % kStages;
      const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
      const int b = it % kAccBufs;
      const uint32_t aph = static_cast<uint32_t>(it / kAccBufs) & 1u;
      if (*abort_flag) break;
      // acc_full: the MMAs are done; full: the producer's writes to the stage
      // (metadata, weights) are visible to this thread.
      const bool got = mbar_wait(&acc_full[b], aph, timeout) && mbar_wait(&full[s], ph, timeout);
      if (!got) fail(abort_flag, kStatusEpilogueWait);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      const uint8_t* st = smem + s * kStageBytes;
      const int4 meta = *reinterpret_cast<const int4*>(st + kOffMeta);
      if (meta.y < 0) break;
      tc_fence_after_sync();
      float v[kRowsB];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(b * kRowsB);
      tmem_ld_32x32b_x32(taddr, v);
      tmem_ld_32x32b_x32(taddr + 32, v + 32);
      tmem_ld_32x32b_x32(taddr + 64, v + 64);
      tmem_ld_32x32b_x32(taddr + 96, v + 96);
      tmem_ld_wait(v);
      tmem_ld_wait(v + 32);
      tmem_ld_wait(v + 64);
      tmem_ld_wait(v + 96);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      const int key = meta.x * kKeysPerTile + quad * 32 + lane;
      // Per token: sum_h w_h max(0, d_h), two heads per packed FMA in four
      // independent chains; the weights are the same for the whole warp
      // (broadcast reads).
      float score[kTokensPerTile];
#pragma unroll
      for (int tok = 0; tok < kTokensPerTile; ++tok) {
        const float4* wv = reinterpret_cast<const float4*>(st + kOffW) + tok * (kNumHeads / 4);
        const float* d = v + tok * kNumHeads;
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};   // packed (+0, +0)
#pragma unroll
        for (int i = 0; i < kNumHeads / 4; ++i) {
          const float4 wq = wv[i];
          acc[i & 3] = f2_fma(f2_pack(fmaxf(d[4 * i], 0.f), fmaxf(d[4 * i + 1], 0.f)), f2_pack(wq.x, wq.y), acc[i & 3]);
          acc[(i + 2) & 3] =
              f2_fma(f2_pack(fmaxf(d[4 * i + 2], 0.f), fmaxf(d[4 * i + 3], 0.f)), f2_pack(wq.z, wq.w), acc[(i + 2) & 3]);
        }
        const uint64_t sum = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
        float lo, hi;
        f2_unpack(sum, lo, hi);
        score[tok] = lo + hi;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);   // this warp is done with the stage
      if (key < meta.z) args.logits[static_cast<long long>(2 * meta.y) * args.ld + key] = score[0];
      if (key < meta.w) args.logits[static_cast<long long>(2 * meta.y + 1) * args.ld + key] = score[1];
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------- top-k

constexpr int kTopkThreads = 256;
constexpr int kTopkCacheMax = 12288;   // rows up to this many keys are read once, into shared memory

// Order-preserving key of a float score (larger score -> larger key); -0 is
// taken as +0 so that the two zeros tie and the smaller index wins.
__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive prefix sum of one value per thread; returns the
// thread's prefix and writes the block total to *total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* scratch, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = lane < kTopkThreads / 32 ? scratch[lane] : 0u;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, t, d);
      if (lane >= d) t += y;
    }
    if (lane < kTopkThreads / 32) scratch[lane] = t;   // inclusive over warps
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? scratch[warp - 1] : 0u;
  *total = scratch[kTopkThreads / 32 - 1];
  __syncthreads();
  return before + x - v;
}

// The digit d (of the histogram's nb bins, largest first) that holds the
// rank-th largest of the counted keys (rank from 1), and *above = the count of
// keys with a larger digit.
__device__ uint32_t find_digit(const uint32_t* hist, int nb, uint32_t rank, uint32_t* scratch, uint32_t* above) {
  __shared__ uint32_t found_digit, found_above;
  const int per = nb / kTopkThreads;
  const int first = nb - (threadIdx.x + 1) * per;   // thread 0 takes the largest digits
  uint32_t run = 0;
  for (int j = 0; j < per; ++j) run += hist[first + j];
  uint32_t total;
  const uint32_t before = block_exclusive_scan(run, scratch, &total);   // keys with larger digits
  if (before < rank && rank <= before + run) {
    uint32_t acc = before;
    for (int j = per - 1; j >= 0; --j) {
      const uint32_t c = hist[first + j];
      if (acc < rank && rank <= acc + c) {
        found_digit = static_cast<uint32_t>(first + j);
        found_above = acc;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
  *above = found_above;
  return found_digit;
}

// K6: per query row t, the k visible keys with the largest scores (see the
// file comment).  Rows of at most kTopkCacheMax visible keys are read from
// global memory once, as order-preserving keys into shared memory; longer
// rows are read again by every pass.
__global__ void __launch_bounds__(kTopkThreads)
    indexer_topk_kernel(const float* __restrict__ logits, long long ld, int N, const int32_t* __restrict__ len,
                        int k, int32_t* __restrict__ out, int cache_keys) {
  extern __shared__ uint32_t cache[];   // cache_keys words
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t scratch[kTopkThreads / 32];
  // The scores are the preceding kernel's output.
  grid_dependency_wait();
  const int t = blockIdx.x;
  const float* row = logits + static_cast<long long>(t) * ld;
  int32_t* dst = out + static_cast<long long>(t) * k;
  int L = len[t];
  L = L < 0 ? 0 : (L > N ? N : L);
  if (L <= k) {
    for (int i = threadIdx.x; i < k; i += kTopkThreads) dst[i] = i < L ? i : -1;
    return;
  }
  const bool cached = L <= cache_keys;
  auto key_at = [&](int i) -> uint32_t { return cached ? cache[i] : score_key(row[i]); };

  // Digit 1: bits 31..21 (read the row, cache it).
  for (int i = threadIdx.x; i < 2048; i += kTopkThreads) hist[i] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < L; i += kTopkThreads) {
    const uint32_t key = score_key(row[i]);
    if (cached) cache[i] = key;
    atomicAdd(&hist[key >> 21], 1u);
  }
  __syncthreads();
  uint32_t above1, above2, above3;
  const uint32_t d1 = find_digit(hist, 2048, static_cast<uint32_t>(k), scratch, &above1);
  // Digit 2: bits 20..10 of the keys with digit 1 = d1.
  for (int i = threadIdx.x; i < 2048; i += kTopkThreads) hist[i] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < L; i += kTopkThreads) {
    const uint32_t key = key_at(i);
    if ((key >> 21) == d1) atomicAdd(&hist[(key >> 10) & 0x7FFu], 1u);
  }
  __syncthreads();
  const uint32_t d2 = find_digit(hist, 2048, static_cast<uint32_t>(k) - above1, scratch, &above2);
  // Digit 3: bits 9..0 of the keys with digits (d1, d2).
  for (int i = threadIdx.x; i < 1024; i += kTopkThreads) hist[i] = 0u;
  __syncthreads();
  const uint32_t hi22 = (d1 << 11) | d2;
  for (int i = threadIdx.x; i < L; i += kTopkThreads) {
    const uint32_t key = key_at(i);
    if ((key >> 10) == hi22) atomicAdd(&hist[key & 0x3FFu], 1u);
  }
  __syncthreads();
  const uint32_t d3 = find_digit(hist, 1024, static_cast<uint32_t>(k) - above1 - above2, scratch, &above3);
  const uint32_t T = (hi22 << 10) | d3;
  const uint32_t n_above = above1 + above2 + above3;            // keys > T
  const uint32_t n_equal = static_cast<uint32_t>(k) - n_above;  // keys == T to take, smallest index first

  // Output: thread i takes the contiguous segment [i seg, (i + 1) seg); one
  // scan of its counts gives where its chosen keys go.
  const int seg = (L + kTopkThreads - 1) / kTopkThreads;
  const int b = threadIdx.x * seg;
  const int e = min(L, b + seg);
  uint32_t gt = 0, eq = 0;
  for (int i = b; i < e; ++i) {
    const uint32_t key = key_at(i);
    gt += key > T ? 1u : 0u;
    eq += key == T ? 1u : 0u;
  }
  uint32_t tot;
  const uint32_t gt_before = block_exclusive_scan(gt, scratch, &tot);
  uint32_t eq_before = block_exclusive_scan(eq, scratch, &tot);
  uint32_t pos = gt_before + min(eq_before, n_equal);
  for (int i = b; i < e; ++i) {
    const uint32_t key = key_at(i);
    if (key > T || (key == T && eq_before < n_equal)) dst[pos++] = i;
    if (key == T) ++eq_before;
  }
}

}  // namespace

cudaError_t indexer_setup_device() {
  const cudaError_t err =
      cudaFuncSetAttribute(indexer_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (err != cudaSuccess) return err;
  return cudaFuncSetAttribute(indexer_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kTopkCacheMax * static_cast<int>(sizeof(uint32_t)));
}

cudaError_t launch_indexer_logits(const CUtensorMap& tm_k, const CUtensorMap& tm_q, const uint8_t* q_sf,
                                  const uint8_t* k_sf, const float* w, const int32_t* len, float* logits, long long ld,
                                  int M, int N, int sm_count, unsigned long long timeout_ns, cudaStream_t stream) {
  IndexerArgs a;
  a.k_sf = reinterpret_cast<const uint32_t*>(k_sf);
  a.q_sf = reinterpret_cast<const uint32_t*>(q_sf);
  a.w = w;
  a.len = len;
  a.logits = logits;
  a.ld = ld;
  a.M = M;
  a.N = N;
  a.key_blocks = (N + kKeysPerTile - 1) / kKeysPerTile;
  a.pairs = (M + 1) / 2;
  a.chunks_per_block = (a.pairs + kChunkPairs - 1) / kChunkPairs;
  a.num_chunks = a.key_blocks * a.chunks_per_block;
  a.timeout_ns = timeout_ns;
  const int grid = a.num_chunks < sm_count ? a.num_chunks : sm_count;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, indexer_logits_kernel, tm_k, tm_q, a);
}

cudaError_t launch_indexer_topk(const float* logits, long long ld, int M, int N, const int32_t* len, int k,
                                int32_t* out, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  // Shared memory for the row cache: enough for N keys, at most the cap
  // (longer rows are streamed from global memory by every pass).
  const int cache_keys = N < kTopkCacheMax ? N : kTopkCacheMax;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M, 1, 1);
  cfg.blockDim = dim3(kTopkThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(N <= kTopkCacheMax ? cache_keys : 0) * sizeof(uint32_t);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, indexer_topk_kernel, logits, ld, N, len, k, out,
                            N <= kTopkCacheMax ? cache_keys : 0);
}

cudaError_t read_indexer_status(uint32_t* flags, bool reset) {
  uint32_t v = 0;
  cudaError_t err = cudaMemcpyFromSymbol(&v, g_iq_status_indexer, sizeof(v));
  if (err != cudaSuccess) return err;
  if (flags) *flags = v;
  if (reset) {
    const uint32_t zero = 0;
    err = cudaMemcpyToSymbol(g_iq_status_indexer, &zero, sizeof(zero));
  }
  return err;
}

}  // namespace iq
