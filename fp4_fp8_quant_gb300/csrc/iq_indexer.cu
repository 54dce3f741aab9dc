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
// tcgen05.mma kind::mxf4 block_scale (E2M1 x E2M1, UE8M0 per 32 K) in its
// CTA-pair form.  The keys are the MMA's M side, 256 per instruction (128 in
// each CTA of the pair); two query tokens x 64 heads are its N side (128),
// one token's heads in each CTA; K = 128 in two MMAs of 64.  Each accumulator
// lane of a CTA is one of its keys and holds all 64 heads of both tokens, so
// the ReLU and the weighted sum over the heads stay inside one thread of the
// epilogue.  Work comes in chunks of one 256-key block and 16 consecutive
// query tokens, tile j pairing tokens j and 8 + j: each CTA's query rows for
// the chunk (8 tokens x 64 heads) are then contiguous and, like the keys, the
// scale words and the weights, are loaded once per chunk into one of three
// slots, so the MMA issuer's per-tile work is two MMAs and a commit.  Warp
// roles (320 threads per CTA): warp 0 stages the slots (TMA with the 64-byte
// swizzle for keys and queries, a bulk copy for the weights, scale words
// transposed through registers into the layout tcgen05.cp reads; one
// cluster-scope arrive per chunk); warp 1 owns tensor memory and, in the
// leader CTA, issues each chunk's scale copies and its tiles' MMAs in order
// into three accumulator buffers; warps 2..9, two groups of four (one warp
// per 32-lane quarter of tensor memory) taking alternate tiles, drain an
// accumulator and form their 32 keys' scores for both tokens.  Chunks are
// dealt to the CTA pairs round robin; tiles whose two tokens see no key of
// the block are skipped.
//
// K6 indexer_topk_kernel.  One CTA per query row: radix selection of the k-th
// largest score over order-preserving 32-bit keys (11, 11, then 10 bits,
// histograms in shared memory; a row of up to 12288 keys is read once and
// kept in shared memory), then a pass in index order over contiguous
// per-thread segments that writes the keys above the threshold and the first
// (smallest-index) keys equal to it.  Every sweep takes four keys per access
// when the row is 16-byte aligned; rows longer than 12288 keys take 1024
// threads and a cache of up to 49152 keys.
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

constexpr int kKeysPerCta = 128;                      // MMA M per CTA
constexpr int kKeysPerTile = 2 * kKeysPerCta;         // 256 keys per pair tile
constexpr int kChunkTokens = 16;                      // query tokens per chunk
constexpr int kHalfTokens = kChunkTokens / 2;         // tile j: tokens j (CTA 0) and 8 + j (CTA 1)
constexpr int kRowsB = 2 * kNumHeads;                 // MMA N = 128
constexpr int kRowBytes = kHeadDim / 2;               // 64: one packed FP4 head / key
constexpr int kKeyTileBytes = kKeysPerCta * kRowBytes;     // 8 KB per CTA
constexpr int kQRows = kHalfTokens * kNumHeads;            // 512 query rows per CTA and chunk
constexpr int kQBoxRows = 256;                             // rows per tensor-map box
constexpr int kQTileBytes = kNumHeads * kRowBytes;         // 4 KB: one token's heads
constexpr int kSlots = 3;                             // chunks in flight
constexpr int kAccBufs = 3;
constexpr int kEpiWarps = 12;                         // three groups of four, tile i to group i % 3
constexpr int kGroupWarps = 4;
constexpr int kEpiGroups = kEpiWarps / kGroupWarps;
static_assert(kEpiGroups == kAccBufs, "each epilogue group drains its own accumulator buffer");
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr uint16_t kPairMask = 0x3;
constexpr uint32_t kTmemCols = 512;
// Scale factors in tensor memory, per slot: the chunk's query scales, 4
// columns per tile (384 + 32 slot + 4 j), and its key scales (480 + 4 slot),
// copied when the chunk's MMAs begin.
constexpr uint32_t kSfbCol = kAccBufs * kRowsB;
constexpr uint32_t kSfaCol = kSfbCol + kSlots * 4 * kHalfTokens;
static_assert(kSfaCol + 4 * kSlots <= kTmemCols, "tensor memory columns");

// A slot holds one chunk: this CTA's query rows (8 tokens x 64 heads, 64-byte
// swizzle), its 128 keys, the key scales and the 8 tiles' query scales (both
// tokens of each, as every CTA's tensor memory holds the scales of all N rows)
// in the tcgen05.cp 32x128b layout, the 16 tokens' weights and the metadata.
constexpr int kSlotQ = 0;
constexpr int kSlotK = kQRows * kRowBytes;
constexpr int kSlotSfa = kSlotK + kKeyTileBytes;
constexpr int kSlotSfb = kSlotSfa + 512;
constexpr int kSlotW = kSlotSfb + kHalfTokens * 512;
constexpr int kSlotMeta = kSlotW + kChunkTokens * kNumHeads * 4;   // int[20]
constexpr int kSlotBytes = 49 * 1024;
static_assert(kSlotMeta + 20 * 4 <= kSlotBytes && kSlotK % 1024 == 0, "slot layout");
constexpr int kOffBar = kSlots * kSlotBytes;
constexpr int kNumBars = 3 * kSlots + 2 * kAccBufs + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // over half of an SM: one CTA per SM
static_assert(kSmemBytes > 114 * 1024 && kSmemBytes <= 227 * 1024, "one CTA per SM");
static_assert(kOffBar + kNumBars * 8 <= kOffMisc, "barriers");
// Metadata: [0] the visible tiles (bits 0-7) or kEndChunk, [1] key block,
// [2] first token, [4 + i] visible length of token i of the chunk.
constexpr int kEndChunk = 1 << 30;

struct IndexerArgs {
  const uint32_t* k_sf;   // [N] scale words (4 UE8M0 bytes per key)
  const uint32_t* q_sf;   // [M * 64] scale words (4 per (token, head))
  const float* w;         // [M][64]
  const int32_t* len;     // [M]
  float* logits;          // [M][ld]
  long long ld;
  int M, N;
  int key_blocks, chunks_per_block, num_chunks;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ void fail(volatile uint32_t* abort_flag, uint32_t bit) {
  atomicOr(&g_iq_status_indexer, bit);
  *abort_flag = 1u;
}

// Length of token i of chunk ch (lanes 0..15), clamped to [0, N]; 0 past M.
__device__ __forceinline__ int chunk_lengths(const IndexerArgs& a, int ch, int lane) {
  if (ch >= a.num_chunks || lane >= kChunkTokens) return 0;
  const int kb = ch / a.chunks_per_block;
  const int t = (ch - kb * a.chunks_per_block) * kChunkTokens + lane;
  if (t >= a.M) return 0;
  const int L = static_cast<int>(ld_dependent_u32(a.len + t));
  return L < 0 ? 0 : (L > a.N ? a.N : L);
}

// Scale words of 128 rows into the tcgen05.cp 32x128b layout (word [r * 4 +
// c] = row c * 32 + r): lane l holds rows 4l..4l+3 in `v`.
__device__ __forceinline__ void store_scale_rows(uint32_t* dst, int lane, const uint4& v) {
  const int c = lane >> 3, r = (lane & 7) * 4;
  dst[(r + 0) * 4 + c] = v.x;
  dst[(r + 1) * 4 + c] = v.y;
  dst[(r + 2) * 4 + c] = v.z;
  dst[(r + 3) * 4 + c] = v.w;
}

// Four consecutive scale words from `src`, of which the first `n` exist.
// The query scales are the preceding kernel's output, so these are loads that
// stay below the dependency wait (not the read-only path, which the compiler
// may hoist above it).
__device__ __forceinline__ uint4 load_scale_words(const uint32_t* src, int n) {
  if (n >= 4) return ld_dependent_v4(src);
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (n > 0) v.x = ld_dependent_u32(src);
  if (n > 1) v.y = ld_dependent_u32(src + 1);
  if (n > 2) v.z = ld_dependent_u32(src + 2);
  return v;
}

__global__ void __launch_bounds__(kThreads, 1)
    indexer_logits_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ IndexerArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* kfull = bars;                         // leader: both CTAs' slots loaded and staged
  uint64_t* kstaged = bars + kSlots;              // this CTA's slot: metadata written, weights landed
  uint64_t* kempty = bars + 2 * kSlots;           // the chunk's MMAs and this CTA's epilogue warps are done
  uint64_t* acc_full = bars + 3 * kSlots;         // accumulator b complete (both CTAs)
  uint64_t* acc_empty = acc_full + kAccBufs;      // leader: the pair's eight epilogue warps drained b
  uint64_t* final_bar = acc_empty + kAccBufs;     // every MMA of the pair completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + 4);
  auto slot_ptr = [&](int k) { return smem + k * kSlotBytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t timeout = args.timeout_ns;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_q);
    for (int k = 0; k < kSlots; ++k) {
      mbar_init(&kfull[k], 3);                    // leader's expect-tx arrive + both CTAs' staging arrives
      mbar_init(&kstaged[k], 1);
      mbar_init(&kempty[k], 1 + kEpiWarps);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 2 * kGroupWarps);
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
  const uint32_t kfull_l0 = mapa_shared(smem_u32(&kfull[0]), 0);
  const uint32_t acc_empty_l0 = mapa_shared(smem_u32(&acc_empty[0]), 0);
  const int pair_id = static_cast<int>(cluster_id_x());
  const int num_pairs = static_cast<int>(cluster_count_x());
  // The queries' FP4 Q may be the preceding kernel's output.  The next
  // kernel (the top-k selection) may be scheduled now: it waits for this
  // one's completion before it reads the scores.
  grid_dependency_wait();
  grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Chunks ch = pair_id, + num_pairs, ... with a visible tile, each into
    // the next slot: the metadata, the scale words (loaded four rows per
    // lane, stored transposed into the tcgen05.cp layout), the weights by a
    // bulk copy on this CTA's slot barrier, the keys and the query rows by
    // TMA on the leader's; then one cluster-scope arrive on the leader's slot
    // barrier.  Last, an end chunk.
    uint32_t issued_mask = 0, issued_phase = 0;
    int nchunk = 0;
    bool ok = true;
    auto next_slot = [&](int& slot, uint32_t& kph) -> bool {
      slot = nchunk % kSlots;
      kph = static_cast<uint32_t>(nchunk / kSlots) & 1u;
      ++nchunk;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&kempty[slot], kph ^ 1u, timeout))) {
        if (lane == 0) fail(abort_flag, kStatusProducerWait);
        return false;
      }
      return true;
    };
    int lv = chunk_lengths(args, pair_id, lane);
    for (int ch = pair_id; ch < args.num_chunks && ok; ch += num_pairs) {
      const int lv_next = chunk_lengths(args, ch + num_pairs, lane);   // in flight during this chunk
      const int kb = ch / args.chunks_per_block;
      const int tb = (ch - kb * args.chunks_per_block) * kChunkTokens;
      uint32_t vis = 0;   // tiles with a token that sees a key of the block (warp-uniform)
#pragma unroll
      for (int j = 0; j < kHalfTokens; ++j) {
        const int L = max(__shfl_sync(0xFFFFFFFFu, lv, j), __shfl_sync(0xFFFFFFFFu, lv, kHalfTokens + j));
        if (kb * kKeysPerTile < L) vis |= 1u << j;
      }
      const int lv_here = lv;
      lv = lv_next;
      if (vis == 0u) continue;
      if (__any_sync(0xFFFFFFFFu, *abort_flag != 0u)) {
        ok = false;
        break;
      }
      int slot;
      uint32_t kph;
      if (!(ok = next_slot(slot, kph))) break;
      uint8_t* ks = slot_ptr(slot);
      int* meta = reinterpret_cast<int*>(ks + kSlotMeta);
      if (lane < kChunkTokens) meta[4 + lane] = lv_here;
      if (lane == 0) {
        meta[0] = static_cast<int>(vis);
        meta[1] = kb;
        meta[2] = tb;
      }
      // Scale words: this CTA's 128 keys, then per visible tile its 128
      // query rows (token tb + j's heads, then token tb + 8 + j's).  Every
      // load goes out before the first store, so the chunk waits for one
      // load latency, not nine.
      uint4 sfw[1 + kHalfTokens];
      {
        const int key0 = kb * kKeysPerTile + static_cast<int>(rank) * kKeysPerCta + 4 * lane;
        sfw[0] = load_scale_words(args.k_sf + (key0 < args.N ? key0 : 0), min(4, args.N - key0));
      }
#pragma unroll
      for (int j = 0; j < kHalfTokens; ++j) {
        const int t = tb + j + (lane >= 16 ? kHalfTokens : 0);
        const bool need = ((vis >> j) & 1u) && t < args.M;
        sfw[1 + j] = load_scale_words(args.q_sf + static_cast<long long>(need ? t : 0) * kNumHeads + 4 * (lane & 15),
                                      need ? 4 : 0);
      }
      store_scale_rows(reinterpret_cast<uint32_t*>(ks + kSlotSfa), lane, sfw[0]);
#pragma unroll
      for (int j = 0; j < kHalfTokens; ++j)
        if ((vis >> j) & 1u) store_scale_rows(reinterpret_cast<uint32_t*>(ks + kSlotSfb + j * 512), lane, sfw[1 + j]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        // Weights of the chunk's tokens that exist (rows past M are never read).
        const uint32_t wbytes = static_cast<uint32_t>(min(kChunkTokens, args.M - tb) * kNumHeads * 4);
        mbar_arrive_expect_tx(&kstaged[slot], wbytes);
        bulk_load(ks + kSlotW, args.w + static_cast<long long>(tb) * kNumHeads, wbytes, &kstaged[slot]);
        if (leader) mbar_arrive_expect_tx(&kfull[slot], 2 * (kKeyTileBytes + kQRows * kRowBytes));
        const uint32_t kbar = kfull_l0 + 8u * static_cast<uint32_t>(slot);
        tma_load_2d_pair(ks + kSlotK, &tm_k, kbar, 0, kb * kKeysPerTile + static_cast<int>(rank) * kKeysPerCta);
        const int qrow0 = (tb + static_cast<int>(rank) * kHalfTokens) * kNumHeads;
        tma_load_2d_pair(ks + kSlotQ, &tm_q, kbar, 0, qrow0);
        tma_load_2d_pair(ks + kSlotQ + kQBoxRows * kRowBytes, &tm_q, kbar, 0, qrow0 + kQBoxRows);
        mbar_arrive_cluster(kbar);   // this CTA's scale words staged
        issued_mask |= 1u << slot;
        issued_phase = (issued_phase & ~(1u << slot)) | (kph << slot);
      }
    }
    // The end chunk: metadata only.
    if (ok) {
      int slot;
      uint32_t kph;
      if (next_slot(slot, kph)) {
        if (lane == 0) {
          reinterpret_cast<volatile int*>(slot_ptr(slot) + kSlotMeta)[0] = kEndChunk;
          mbar_arrive(&kstaged[slot]);
          if (leader) mbar_arrive(&kfull[slot]);
          mbar_arrive_cluster(kfull_l0 + 8u * static_cast<uint32_t>(slot));
        }
      }
    }
    // Teardown: the pair's MMAs read this CTA's slots; wait (bounded) until
    // every loaded slot was released.
    if (lane == 0) {
      for (int k = 0; k < kSlots; ++k)
        if (((issued_mask >> k) & 1u) && !mbar_wait(&kempty[k], (issued_phase >> k) & 1u, 2 * timeout))
          fail(abort_flag, kStatusTeardownWait);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------- MMA issuer (leader)
    // Chunk by chunk: the scale copies, then per visible tile two MMAs into
    // the next accumulator buffer; the slot is released after the chunk's
    // last MMAs.
    if (lane == 0) {
      if (leader) {
        const uint32_t idesc_k0 = idesc_mxf4_e2m1(kKeysPerTile, kRowsB, 0, 0);
        const uint32_t idesc_k1 = idesc_mxf4_e2m1(kKeysPerTile, kRowsB, 2, 2);
        int it = 0;
        for (int n = 0;; ++n) {
          const int slot = n % kSlots;
          if (*abort_flag) break;
          if (!mbar_wait(&kfull[slot], static_cast<uint32_t>(n / kSlots) & 1u, timeout)) {
            fail(abort_flag, kStatusMmaWait);
            break;
          }
          tc_fence_after_sync();
          const uint8_t* ks = slot_ptr(slot);
          const int vis = reinterpret_cast<const volatile int*>(ks + kSlotMeta)[0];
          if (vis & kEndChunk) break;
          const uint32_t sfa = tmem + kSfaCol + 4u * static_cast<uint32_t>(slot);
          const uint32_t sfb0 = tmem + kSfbCol + 4u * kHalfTokens * static_cast<uint32_t>(slot);
          tc_cp_32x128b_warpx4_pair(sfa, smem_desc_sf(smem_u32(ks + kSlotSfa)));
          for (int j = 0; j < kHalfTokens; ++j)
            if ((vis >> j) & 1)
              tc_cp_32x128b_warpx4_pair(sfb0 + 4u * j, smem_desc_sf(smem_u32(ks + kSlotSfb + j * 512)));
          const uint64_t adesc = smem_desc_sw64(smem_u32(ks + kSlotK));
          bool ok = true;
          for (int j = 0; j < kHalfTokens && ok; ++j) {
            if (!((vis >> j) & 1)) continue;
            const int b = it % kAccBufs;
            const uint32_t aph = static_cast<uint32_t>(it / kAccBufs) & 1u;
            ++it;
            if (!mbar_wait(&acc_empty[b], aph ^ 1u, timeout)) {
              fail(abort_flag, kStatusMmaWait);
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint64_t bdesc = smem_desc_sw64(smem_u32(ks + kSlotQ + j * kQTileBytes));
            const uint32_t d = tmem + static_cast<uint32_t>(b * kRowsB);
            const uint32_t sfb = sfb0 + 4u * static_cast<uint32_t>(j);
            // K = 128: dims 0..63 (scale bytes 0, 1), then dims 64..127 (bytes
            // 2, 3), 32 bytes further along each 64-byte row.
            tc_mma_mxf4_pair(d, adesc, bdesc, idesc_k0, sfa, sfb, 0u);
            tc_mma_mxf4_pair(d, adesc + 2, bdesc + 2, idesc_k1, sfa, sfb, 1u);
            tc_commit_pair(&acc_full[b], kPairMask);
          }
          if (!ok) break;
          tc_commit_pair(&kempty[slot], kPairMask);
        }
        tc_commit_pair(final_bar, kPairMask);
      }
      // Both CTAs: every pair MMA that uses this CTA's memory has completed.
      if (!mbar_wait(final_bar, 0, 2 * timeout)) fail(abort_flag, kStatusTeardownWait);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // The same chunk walk; group (warp - 2) / 4 takes visible tile i
    // (counted over all chunks) when i % 3 is its index, and with it
    // accumulator buffer i % 3; each warp drains TMEM lanes 32 quad ..
    // 32 quad + 31 (32 keys), one token (64 columns) at a time; after a chunk
    // every warp releases the slot.
    const int quad = warp & 3;
    const int group = (warp - 2) >> 2;
    int it = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int slot = n % kSlots;
      if (*abort_flag) break;
      const bool got = mbar_wait(&kstaged[slot], static_cast<uint32_t>(n / kSlots) & 1u, timeout);
      if (!got) fail(abort_flag, kStatusEpilogueWait);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      const uint8_t* ks = slot_ptr(slot);
      const int* meta = reinterpret_cast<const int*>(ks + kSlotMeta);
      const int vis = meta[0];
      if (vis & kEndChunk) break;
      const int kb = meta[1], tb = meta[2];
      const int key = kb * kKeysPerTile + static_cast<int>(rank) * kKeysPerCta + quad * 32 + lane;
      for (int j = 0; j < kHalfTokens; ++j) {
        if (!((vis >> j) & 1)) continue;
        const int b = it % kAccBufs;
        const uint32_t aph = static_cast<uint32_t>(it / kAccBufs) & 1u;
        const bool mine = b == group;
        ++it;
        if (!mine) continue;
        const bool acc = mbar_wait(&acc_full[b], aph, timeout);
        if (!acc) fail(abort_flag, kStatusEpilogueWait);
        if (!__all_sync(0xFFFFFFFFu, acc)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(b * kRowsB);
        // Per token: sum_h w_h max(0, d_h), two heads per packed FMA in four
        // independent chains; the weights are the same for the whole warp
        // (broadcast reads).  Columns 0..63: token tb + j; 64..127: tb + 8 + j.
        // The accumulator is released once the second token's columns are in
        // registers.
        float score[2];
#pragma unroll
        for (int tok = 0; tok < 2; ++tok) {
          float d[kNumHeads];
          tmem_ld_32x32b_x32(taddr + tok * kNumHeads, d);
          tmem_ld_32x32b_x32(taddr + tok * kNumHeads + 32, d + 32);
          tmem_ld_wait(d);
          tmem_ld_wait(d + 32);
          if (tok == 1) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(acc_empty_l0 + 8u * static_cast<uint32_t>(b));
          }
          const float4* wv = reinterpret_cast<const float4*>(ks + kSlotW) + (j + tok * kHalfTokens) * (kNumHeads / 4);
          uint64_t accv[4] = {0ull, 0ull, 0ull, 0ull};   // packed (+0, +0)
#pragma unroll
          for (int i = 0; i < kNumHeads / 4; ++i) {
            const float4 wq = wv[i];
            accv[i & 3] =
                f2_fma(f2_pack(fmaxf(d[4 * i], 0.f), fmaxf(d[4 * i + 1], 0.f)), f2_pack(wq.x, wq.y), accv[i & 3]);
            accv[(i + 2) & 3] = f2_fma(f2_pack(fmaxf(d[4 * i + 2], 0.f), fmaxf(d[4 * i + 3], 0.f)),
                                       f2_pack(wq.z, wq.w), accv[(i + 2) & 3]);
          }
          const uint64_t sum = f2_add(f2_add(accv[0], accv[1]), f2_add(accv[2], accv[3]));
          float lo, hi;
          f2_unpack(sum, lo, hi);
          score[tok] = lo + hi;
        }
        const int L0 = meta[4 + j], L1 = meta[4 + kHalfTokens + j];
        if (key < L0) args.logits[static_cast<long long>(tb + j) * args.ld + key] = score[0];
        if (key < L1) args.logits[static_cast<long long>(tb + kHalfTokens + j) * args.ld + key] = score[1];
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&kempty[slot]);   // this warp is done with the slot
    }
  }

  // Neither CTA leaves (or frees tensor memory) while the pair may still use
  // its shared memory, barriers or tensor memory.
  tc_fence_before_sync();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------- top-k

constexpr int kTopkThreads = 256;
constexpr int kTopkLongThreads = 1024;   // rows longer than the cache
constexpr int kTopkLongCacheMax = 49152;   // the 1024-thread instance's row cache (192 KB, one CTA per SM)
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
template <int kThreads>
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
    uint32_t t = lane < kThreads / 32 ? scratch[lane] : 0u;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, t, d);
      if (lane >= d) t += y;
    }
    if (lane < kThreads / 32) scratch[lane] = t;   // inclusive over warps
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? scratch[warp - 1] : 0u;
  *total = scratch[kThreads / 32 - 1];
  __syncthreads();
  return before + x - v;
}

// The digit d (of the histogram's nb bins, largest first) that holds the
// rank-th largest of the counted keys (rank from 1), and *above = the count of
// keys with a larger digit.
template <int kThreads>
__device__ uint32_t find_digit(const uint32_t* hist, int nb, uint32_t rank, uint32_t* scratch, uint32_t* above) {
  __shared__ uint32_t found_digit, found_above;
  const int per = nb / kThreads;
  const int first = nb - (threadIdx.x + 1) * per;   // thread 0 takes the largest digits
  uint32_t run = 0;
  for (int j = 0; j < per; ++j) run += hist[first + j];
  uint32_t total;
  const uint32_t before = block_exclusive_scan<kThreads>(run, scratch, &total);   // keys with larger digits
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
// file comment).  Rows of at most cache_keys visible keys are read from
// global memory once, as order-preserving keys into shared memory; longer
// rows are read again by every pass.  Two instances: 256 threads with a cache
// of up to kTopkCacheMax keys (eight CTAs per SM), and, when the rows can be
// longer than that, 1024 threads with a cache of up to kTopkLongCacheMax.
template <int kThreads>
__global__ void __launch_bounds__(kThreads, 2048 / kThreads)
    indexer_topk_kernel(const float* logits, long long ld, int N, const int32_t* len, int k,
                        int32_t* __restrict__ out, int cache_keys) {
  // Both are read and written with 16-byte accesses.
  extern __shared__ __align__(16) uint32_t cache[];   // cache_keys words
  __shared__ __align__(16) uint32_t hist[2048];
  __shared__ uint32_t scratch[kThreads / 32];
  // The scores are the preceding kernel's output.  They and the lengths are
  // read through plain pointers (no __restrict__, no read-only path), so the
  // compiler keeps those loads below the wait.
  grid_dependency_wait();
  const int t = blockIdx.x;
  const float* row = logits + static_cast<long long>(t) * ld;
  int32_t* dst = out + static_cast<long long>(t) * k;
  int L = len[t];
  L = L < 0 ? 0 : (L > N ? N : L);
  if (L <= k) {
    for (int i = threadIdx.x; i < k; i += kThreads) dst[i] = i < L ? i : -1;
    return;
  }
  const bool cached = L <= cache_keys;
  auto key_at = [&](int i) -> uint32_t { return cached ? cache[i] : score_key(row[i]); };
  // Four keys per access where the row is 16-byte aligned (16-byte loads of
  // the scores and of the cache); the last L % 4 keys, or every key of an
  // unaligned row, one at a time.  Every pass visits each key exactly once.
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0u;
  const int L4 = vec ? L >> 2 : 0;
  auto quad_at = [&](int q) -> uint4 {
    if (cached) return reinterpret_cast<const uint4*>(cache)[q];
    const float4 f = reinterpret_cast<const float4*>(row)[q];
    return make_uint4(score_key(f.x), score_key(f.y), score_key(f.z), score_key(f.w));
  };
  auto for_each_key = [&](auto&& fn) {
    for (int q = threadIdx.x; q < L4; q += kThreads) {
      const uint4 kk = quad_at(q);
      fn(kk.x);
      fn(kk.y);
      fn(kk.z);
      fn(kk.w);
    }
    for (int i = 4 * L4 + threadIdx.x; i < L; i += kThreads) fn(key_at(i));
  };

  // Digit 1: bits 31..21 (read the row, cache it).
  for (int i = threadIdx.x; i < 2048; i += kThreads) hist[i] = 0u;
  __syncthreads();
  for (int q = threadIdx.x; q < L4; q += kThreads) {
    const float4 f = reinterpret_cast<const float4*>(row)[q];
    const uint4 kk = make_uint4(score_key(f.x), score_key(f.y), score_key(f.z), score_key(f.w));
    if (cached) reinterpret_cast<uint4*>(cache)[q] = kk;
    atomicAdd(&hist[kk.x >> 21], 1u);
    atomicAdd(&hist[kk.y >> 21], 1u);
    atomicAdd(&hist[kk.z >> 21], 1u);
    atomicAdd(&hist[kk.w >> 21], 1u);
  }
  for (int i = 4 * L4 + threadIdx.x; i < L; i += kThreads) {
    const uint32_t key = score_key(row[i]);
    if (cached) cache[i] = key;
    atomicAdd(&hist[key >> 21], 1u);
  }
  __syncthreads();
  uint32_t above1, above2, above3;
  const uint32_t d1 = find_digit<kThreads>(hist, 2048, static_cast<uint32_t>(k), scratch, &above1);
  // Digit 2: bits 20..10 of the keys with digit 1 = d1.
  for (int i = threadIdx.x; i < 2048; i += kThreads) hist[i] = 0u;
  __syncthreads();
  for_each_key([&](uint32_t key) {
    if ((key >> 21) == d1) atomicAdd(&hist[(key >> 10) & 0x7FFu], 1u);
  });
  __syncthreads();
  const uint32_t d2 = find_digit<kThreads>(hist, 2048, static_cast<uint32_t>(k) - above1, scratch, &above2);
  // Digit 3: bits 9..0 of the keys with digits (d1, d2).
  for (int i = threadIdx.x; i < 1024; i += kThreads) hist[i] = 0u;
  __syncthreads();
  const uint32_t hi22 = (d1 << 11) | d2;
  for_each_key([&](uint32_t key) {
    if ((key >> 10) == hi22) atomicAdd(&hist[key & 0x3FFu], 1u);
  });
  __syncthreads();
  const uint32_t d3 = find_digit<kThreads>(hist, 1024, static_cast<uint32_t>(k) - above1 - above2, scratch, &above3);
  const uint32_t T = (hi22 << 10) | d3;
  const uint32_t n_above = above1 + above2 + above3;            // keys > T
  const uint32_t n_equal = static_cast<uint32_t>(k) - n_above;  // keys == T to take, smallest index first

  // Output: thread i takes the contiguous segment [i seg, (i + 1) seg) (seg a
  // multiple of 4 when the row is aligned); one scan of its counts gives
  // where its chosen keys go.
  const int seg = vec ? ((L + 4 * kThreads - 1) / (4 * kThreads)) * 4 : (L + kThreads - 1) / kThreads;
  const int b = threadIdx.x * seg;
  const int e = min(L, b + seg);
  uint32_t gt = 0, eq = 0;
  auto count = [&](uint32_t key) {
    gt += key > T ? 1u : 0u;
    eq += key == T ? 1u : 0u;
  };
  int i0 = b;
  if (vec) {
    for (; i0 + 4 <= e; i0 += 4) {
      const uint4 kk = quad_at(i0 >> 2);
      count(kk.x);
      count(kk.y);
      count(kk.z);
      count(kk.w);
    }
  }
  for (int i = i0; i < e; ++i) count(key_at(i));
  uint32_t tot;
  const uint32_t gt_before = block_exclusive_scan<kThreads>(gt, scratch, &tot);
  uint32_t eq_before = block_exclusive_scan<kThreads>(eq, scratch, &tot);
  uint32_t pos = gt_before + min(eq_before, n_equal);
  // The chosen indices (exactly k of them, positions 0..k-1) are written to
  // the histogram buffer, free since the last digit was found, and leave in
  // coalesced stores; with k > 2048 they go straight to their destination.
  const bool staged = k <= 2048;
  int32_t* sel = staged ? reinterpret_cast<int32_t*>(hist) : dst;
  auto emit = [&](uint32_t key, int i) {
    if (key > T || (key == T && eq_before < n_equal)) sel[pos++] = i;
    if (key == T) ++eq_before;
  };
  i0 = b;
  if (vec) {
    for (; i0 + 4 <= e; i0 += 4) {
      const uint4 kk = quad_at(i0 >> 2);
      emit(kk.x, i0);
      emit(kk.y, i0 + 1);
      emit(kk.z, i0 + 2);
      emit(kk.w, i0 + 3);
    }
  }
  for (int i = i0; i < e; ++i) emit(key_at(i), i);
  if (staged) {
    __syncthreads();
    if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0u && (k & 3) == 0) {
      for (int q = threadIdx.x; q < (k >> 2); q += kThreads)
        reinterpret_cast<int4*>(dst)[q] = reinterpret_cast<const int4*>(hist)[q];
    } else {
      for (int i = threadIdx.x; i < k; i += kThreads) dst[i] = static_cast<int32_t>(hist[i]);
    }
  }
}

}  // namespace

// Clusters of two (the MMA's CTA pairs), plus programmatic stream
// serialization: the kernel may start while the preceding kernel (the one
// that wrote the queries) runs; it waits for it before reading anything.
cudaLaunchConfig_t logits_config(int pairs, cudaLaunchAttribute* attr, cudaStream_t stream) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// CTA pairs of the logits kernel that fit at once, per device (set-up).
constexpr int kMaxIndexerDevices = 64;
int g_indexer_max_pairs[kMaxIndexerDevices] = {};

int* indexer_pairs_slot() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxIndexerDevices) return nullptr;
  return &g_indexer_max_pairs[dev];
}

cudaError_t indexer_setup_device() {
  cudaError_t err =
      cudaFuncSetAttribute(indexer_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(indexer_topk_kernel<kTopkThreads>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTopkCacheMax * static_cast<int>(sizeof(uint32_t)));
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(indexer_topk_kernel<kTopkLongThreads>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTopkLongCacheMax * static_cast<int>(sizeof(uint32_t)));
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = logits_config(1, attr, nullptr);
  int pairs = 0;
  err = cudaOccupancyMaxActiveClusters(&pairs, indexer_logits_kernel, &cfg);
  if (err != cudaSuccess) return err;
  int* slot = indexer_pairs_slot();
  if (pairs < 1 || slot == nullptr) return cudaErrorInvalidConfiguration;
  *slot = pairs;
  return cudaSuccess;
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
  a.chunks_per_block = (M + kChunkTokens - 1) / kChunkTokens;
  a.num_chunks = a.key_blocks * a.chunks_per_block;
  a.timeout_ns = timeout_ns;
  (void)sm_count;
  const int* slot = indexer_pairs_slot();
  if (slot == nullptr || *slot < 1) return cudaErrorInitializationError;
  const int pairs = a.num_chunks < *slot ? a.num_chunks : *slot;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = logits_config(pairs, attr, stream);
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
  cfg.dynamicSmemBytes = static_cast<size_t>(N <= kTopkCacheMax ? cache_keys : 0) * sizeof(uint32_t);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (N > kTopkCacheMax) {
    // Long rows: four times the threads per row (four times the loads in
    // flight) and a row cache of up to kTopkLongCacheMax keys; longer rows
    // are streamed from global memory by every pass.
    const int long_cache = N <= kTopkLongCacheMax ? N : 0;
    cfg.blockDim = dim3(kTopkLongThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(long_cache) * sizeof(uint32_t);
    return cudaLaunchKernelEx(&cfg, indexer_topk_kernel<kTopkLongThreads>, logits, ld, N, len, k, out, long_cache);
  }
  cfg.blockDim = dim3(kTopkThreads, 1, 1);
  return cudaLaunchKernelEx(&cfg, indexer_topk_kernel<kTopkThreads>, logits, ld, N, len, k, out, cache_keys);
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
