// Internal declarations shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace iq {

// Tiny-amax floor of both block quantizers (the "tiny-scale floor" of the
// TokenSpeed PR, Risk and fallback): blocks whose largest magnitude is below it
// take the scale exponent of the floor.
constexpr float kAmaxFloor = 1e-4f;

constexpr int kLatentDim = 1536;
constexpr int kNumHeads = 64;
constexpr int kHeadDim = 128;
constexpr int kQDim = kNumHeads * kHeadDim;   // 8192
constexpr int kNumKBlocks = kLatentDim / 128; // 12
constexpr int kScaleGroups = kNumKBlocks / 4; // 3 packed int32 words per row
constexpr int kSmallMMax = 128;               // most tokens the small-M kernel takes

// FP4 output variants (compile-time parameter of the fused GEMM kernels).
//   kFp4Mx:    1x32 blocks, UE8M0 scale 2^e with e the smallest integer with
//              6 * 2^e >= amax (never saturates);
//   kFp4MxOcp: 1x32 blocks, UE8M0 scale 2^(floor(log2 amax) - 2) (OCP MX rule,
//              elements saturate at 6);
//   kFp4Nv:    1x16 blocks, E4M3 scale = round-to-nearest of amax / 6 (2^-9 if
//              that is zero), codes of z * (1 / scale).
enum Fp4Format : int { kFp4Mx = 0, kFp4MxOcp = 1, kFp4Nv = 2 };

template <int kFmt>
struct Fp4Layout {
  static constexpr int kBlock = kFmt == kFp4Nv ? 16 : 32;   // elements per scale
  static constexpr int kBlocksPerHead = kHeadDim / kBlock;  // scale bytes per (token, head)
  static constexpr int kScaleBytesPerToken = kQDim / kBlock;
};

// RoPE frequencies of the 32 NeoX pairs, in turns per position unit:
// 10000^(-i/32) / (2 pi), split into a float32 head and tail.
struct RopeTurns {
  float hi[32];
  float lo[32];
};

// Most CTAs a fused-quantizer launch may have (progress flags in the workspace).
constexpr int kMaxFusedCtas = 512;

// Pair-tile orders of the CTA-pair kernel (GemmArgs::order).
constexpr int kOrderFeatureMajor = 0;   // contiguous runs, consecutive tiles share heads
constexpr int kOrderTokenMajor = 1;     // contiguous runs, consecutive tiles share token rows
constexpr int kOrderInterleaved = 2;    // token-major tiles dealt round-robin to the pairs

struct GemmArgs {
  const int32_t* x_sf;   // [3][m_al] packed UE8M0 words of the FP8 latent
  const uint8_t* w_sf;   // [64][12] UE8M0 bytes of the weight blocks
  const int32_t* pos;    // [M]
  uint8_t* q_fp4;        // [M][4096]
  uint8_t* q_sf;         // [M][Fp4Layout<format>::kScaleBytesPerToken]
  float* q_pre;          // [M][8192] or nullptr
  int M;
  int m_al;
  int num_m_tiles;
  int num_m_pairs;       // ceil(num_m_tiles / 2): 256-token row blocks of a CTA pair
  int num_pair_tiles;    // num_m_pairs * (8192 / tile width) pair tiles
  int order;             // pair-tile order: kOrderFeatureMajor, kOrderTokenMajor, kOrderInterleaved
  unsigned long long timeout_ns;
  RopeTurns rope;
  // The quantizer fused into the CTA-pair kernel (interleaved order only):
  // the kernel itself writes the FP8 rows and scale words that it reads
  // through tm_x and x_sf, and counts finished work per 128-row block.
  const uint16_t* latent;        // [M][1536] BF16 bits
  uint8_t* x_fp8;                // [M][1536] E4M3 codes (tm_x's memory)
  int32_t* x_sf_out;             // [3][m_al] packed words (x_sf's memory)
  unsigned long long* ready;     // [1 + kMaxFusedCtas] epoch and per-CTA progress flags, see iq_gemm.cu
  unsigned long long quant_delay_ns;   // diagnostics: delay before each wave's signal
};

// Status bits of the device status word (which wait gave up).
enum : uint32_t {
  kStatusProducerWait = 1u << 0,
  kStatusMmaWait = 1u << 1,
  kStatusEpilogueWait = 1u << 2,
  kStatusTeardownWait = 1u << 3,
  kStatusRowsWait = 1u << 4,     // fused quantizer: token rows not ready in time
};

cudaError_t launch_quant_1x128(const void* x, int M, int K, long long ldx, void* y, long long ldy, int32_t* sf,
                               cudaStream_t stream);

// The quantizer with the lane map for rows in page-locked host memory: the
// same codes and scales; it also copies the M int32 positions pos_src ->
// pos_dst, and max_blocks > 0 caps its grid (the warps then loop).
cudaError_t launch_quant_1x128_host_rows(const void* x, int M, int K, long long ldx, void* y, long long ldy,
                                         int32_t* sf, const int32_t* pos_src, int32_t* pos_dst, int max_blocks,
                                         cudaStream_t stream);

// The FP4 stage's float -> E2M1 conversion alone, one code per byte; n % 8 == 0.
cudaError_t launch_e2m1_codes(const float* x, long long n, uint8_t* codes, cudaStream_t stream);

// Kernel attribute set-up of the fused GEMM on the current device; returns
// how many of its CTA pairs fit on the device at once.
cudaError_t gemm_setup_device(int* max_pairs);
int gemm_pair_size();

// tile_n: output features per pair tile, 256 (two heads) or 128 (one head);
// the W tensor map's box is tile_n / 2 rows.
cudaError_t launch_gemm_rope_hadamard_fp4(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const CUtensorMap& tm_q,
                                          const GemmArgs& args, int tile_n, int fp4_format, int max_pairs,
                                          cudaStream_t stream);

// The same kernel with the quantizer fused in (two-head tiles, interleaved
// order; args.latent, x_fp8, x_sf_out and ready set): one launch for the whole
// preparation.  All CTAs run at once (a cooperative launch).
cudaError_t launch_gemm_fused_quant(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const CUtensorMap& tm_q,
                                    const GemmArgs& args, int fp4_format, int max_pairs, cudaStream_t stream);

// The fused GEMM kernel's wait self-test instance (no TMA loads: every wait
// that depends on them gives up after args.timeout_ns).
cudaError_t launch_gemm_wait_selftest(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const CUtensorMap& tm_q,
                                      const GemmArgs& args, int max_pairs, cudaStream_t stream);

// The small-M (swapped-operand) kernel: M <= kSmallMMax tokens, one launch
// of 64 clusters of two CTAs (one per K half); 64 or 128 token columns.
cudaError_t small_m_setup_device();
cudaError_t launch_small_m_rope_hadamard_fp4(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const GemmArgs& args,
                                             int fp4_format, cudaStream_t stream);

// Device status words of the large-M and small-M kernels (synchronous).
cudaError_t read_device_status(uint32_t* flags, bool reset);
cudaError_t read_small_m_status(uint32_t* flags, bool reset);

// The downstream indexer: scores of (query, key) pairs and top-k selection.
// q_fp4 / k_fp4 are read through the tensor maps tm_q ([M * 64, 64] bytes)
// and tm_k ([N, 64] bytes), 64-byte boxes of 128 rows, 64-byte swizzle.
cudaError_t indexer_setup_device();
cudaError_t launch_indexer_logits(const CUtensorMap& tm_k, const CUtensorMap& tm_q, const uint8_t* q_sf,
                                  const uint8_t* k_sf, const float* w, const int32_t* len, float* logits, long long ld,
                                  int M, int N, int sm_count, unsigned long long timeout_ns, cudaStream_t stream);
cudaError_t launch_indexer_topk(const float* logits, long long ld, int M, int N, const int32_t* len, int k,
                                int32_t* out, cudaStream_t stream);
cudaError_t read_indexer_status(uint32_t* flags, bool reset);

}  // namespace iq
