// C-ABI entry points of the indexer-Q preparation library (include/iq.h):
// argument checks, per-device set-up, TMA descriptor encoding and launches.
// Nothing here allocates device memory; only the diagnostics
// (iq_device_status, iq_selftest_wait_timeout) synchronize.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "iq.h"
#include "iq_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr uint64_t kMaxQuantDelayNs = 1000000ull;   // diagnostics: at most 1 ms per wave

struct DeviceInfo {
  bool ready = false;
  iq_status status = IQ_OK;
  int max_pairs = 0;   // co-resident CTA pairs of the fused GEMM kernel
  int sm_count = 0;
};

std::mutex g_setup_mutex;
DeviceInfo g_devices[kMaxDevices];
std::atomic<int> g_fail_setups{0};   // test hook: set-ups to fail on purpose
std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<int> g_small_m_max{iq::kSmallMMax};
std::atomic<int> g_tile_n_override{0};   // 0: by token count; else 128 or 256
std::atomic<int> g_order_override{0};    // 0: default; 1 feature-major; 2 token-major; 3 interleaved

// Tile width and order of the CTA-pair kernel.  Measured on GB300: up to
// 256 tokens (one 256-row block) the one-head tile spreads the work over 64
// pairs instead of 32 and is faster per call when calls run back to back
// (10.2 against 11.7 us at 128 tokens, 10.6 against 11.8 at 256, inside CUDA
// graphs); from 512 tokens the two-head tile is faster (up to 1.7x at large
// M, where the one-head tile moves half again as many operand bytes from L2
// per FLOP).  Token-major order is as fast or faster at every size, by 4 % at
// 4632 tokens and 16 % at 65536.
int gemm_tile_n(int M) {
  const int o = g_tile_n_override.load(std::memory_order_relaxed);
  if (o == 128 || o == 256) return o;
  return M <= 256 ? 128 : 256;
}

int gemm_order(int) {
  switch (g_order_override.load(std::memory_order_relaxed)) {
    case 1: return iq::kOrderFeatureMajor;
    case 3: return iq::kOrderInterleaved;
    default: return iq::kOrderTokenMajor;
  }
}
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// First call on a device: check the architecture, set kernel attributes and
// resolve the driver's tensor-map encoder.  Success and a wrong architecture
// are cached (later calls only read the cache); a failed CUDA call is not, so
// the next call tries again (a transient failure, e.g. a first call made
// while the stream is being captured, does not disable the device for good).
iq_status device_setup(int* max_pairs, int* sm_count = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return IQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0, pairs = 0;
    iq_status status = IQ_OK;
    if (g_fail_setups.load() > 0) {
      g_fail_setups.fetch_sub(1);
      status = IQ_ERR_CUDA;
    } else if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
               cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      status = IQ_ERR_CUDA;
    } else if (major != 10 || minor != 3) {
      status = IQ_ERR_ARCH;
    } else if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      status = IQ_ERR_CUDA;
    } else if (iq::gemm_setup_device(&pairs) != cudaSuccess || pairs < 1 ||
               iq::small_m_setup_device() != cudaSuccess || iq::indexer_setup_device() != cudaSuccess) {
      status = IQ_ERR_CUDA;
    }
    if (status == IQ_OK && g_encode_tiled == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr) {
        status = IQ_ERR_CUDA;
      } else {
        g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
    }
    if (status == IQ_ERR_CUDA) {
      (void)cudaGetLastError();   // reset the runtime's last-error state for the retry
      return status;
    }
    d.sm_count = sms;
    d.max_pairs = pairs;
    d.status = status;
    d.ready = true;
  }
  *max_pairs = d.max_pairs;
  if (sm_count) *sm_count = d.sm_count;
  return d.status;
}

// 2D uint8 tensor map over a row-major [rows][inner] byte matrix.
bool encode_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                  uint32_t box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

iq::RopeTurns make_rope_turns() {
  iq::RopeTurns t;
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < 32; ++i) {
    const double g = std::pow(10000.0, -static_cast<double>(i) / 32.0) / two_pi;
    t.hi[i] = static_cast<float>(g);
    t.lo[i] = static_cast<float>(g - static_cast<double>(t.hi[i]));
  }
  return t;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace of iq_prepare_q: the FP8 latent [M][1536], its packed scale
// words [3][align4(M)], then the fused quantizer's flags (an epoch word and
// one progress word per CTA, 8 bytes each), each region 256-byte aligned.
size_t prepare_scales_offset(int M) { return align_up(static_cast<size_t>(M) * iq::kLatentDim, 256); }
size_t prepare_counters_offset(int M) {
  return align_up(prepare_scales_offset(M) +
                      static_cast<size_t>(iq::kScaleGroups) * align_up(static_cast<size_t>(M), 4) * sizeof(int32_t),
                  256);
}

// The quantizer fused into the CTA-pair kernel.  Off by default: measured on
// GB300 the fused launch is slower than the two-launch chain at every token
// count (76 against 50 us at 4632 tokens): the quantizing epilogue warps
// become the pipeline's bottleneck and the first MMAs wait for the first
// wave's rows.  On runs the fused launch (tests, measurements).
std::atomic<int> g_quant_fusion{0};
std::atomic<unsigned long long> g_quant_delay_ns{0};

struct FusedQuant {
  const void* latent;
  unsigned long long* counters;
};

iq_status gemm_stage(const void* xq, const int32_t* x_sf, int M, const void* wq, const uint8_t* wq_sf,
                     const int32_t* positions, uint8_t* q_fp4, uint8_t* q_sf, float* q_pre, int fmt, int max_pairs,
                     cudaStream_t stream, const FusedQuant* fuse = nullptr) {
  static const iq::RopeTurns rope = make_rope_turns();
  iq::GemmArgs a{};
  a.x_sf = x_sf;
  a.w_sf = wq_sf;
  a.pos = positions;
  a.q_fp4 = q_fp4;
  a.q_sf = q_sf;
  a.q_pre = q_pre;
  a.M = M;
  a.m_al = (M + 3) / 4 * 4;
  a.num_m_tiles = (M + 127) / 128;
  a.num_m_pairs = (a.num_m_tiles + iq::gemm_pair_size() - 1) / iq::gemm_pair_size();
  const int tile_n = fuse != nullptr ? 256 : gemm_tile_n(M);   // the fused instance has two-head tiles
  a.num_pair_tiles = a.num_m_pairs * (iq::kQDim / tile_n);
  a.order = gemm_order(M);
  a.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  a.rope = rope;
  CUtensorMap tm_x, tm_w, tm_q;
  if (M <= g_small_m_max.load(std::memory_order_relaxed)) {
    // Small-M route: the M token rows per K-block (a box of exactly M rows);
    // one head (128 rows) of W per CTA.
    if (!encode_2d_u8(&tm_x, xq, iq::kLatentDim, static_cast<uint64_t>(M), 128, static_cast<uint32_t>(M)) ||
        !encode_2d_u8(&tm_w, wq, iq::kLatentDim, iq::kQDim, 128, iq::kHeadDim)) {
      return IQ_ERR_CUDA;
    }
    return iq::launch_small_m_rope_hadamard_fp4(tm_x, tm_w, a, fmt, stream) == cudaSuccess ? IQ_OK : IQ_ERR_CUDA;
  }
  // X: this CTA's 128 token rows per K-block; W: half of the tile's W rows
  // per CTA of the pair; Q codes: one head of 128 rows x 64 bytes per store.
  if (!encode_2d_u8(&tm_x, xq, iq::kLatentDim, static_cast<uint64_t>(M), 128, 128) ||
      !encode_2d_u8(&tm_w, wq, iq::kLatentDim, iq::kQDim, 128,
                    static_cast<uint32_t>(tile_n / iq::gemm_pair_size())) ||
      !encode_2d_u8(&tm_q, q_fp4, iq::kQDim / 2, static_cast<uint64_t>(M), 64, 128, CU_TENSOR_MAP_SWIZZLE_64B)) {
    return IQ_ERR_CUDA;
  }
  if (fuse != nullptr) {
    a.order = iq::kOrderInterleaved;
    a.latent = static_cast<const uint16_t*>(fuse->latent);
    a.x_fp8 = static_cast<uint8_t*>(const_cast<void*>(xq));
    a.x_sf_out = const_cast<int32_t*>(x_sf);
    a.ready = fuse->counters;
    a.quant_delay_ns = g_quant_delay_ns.load(std::memory_order_relaxed);
    return iq::launch_gemm_fused_quant(tm_x, tm_w, tm_q, a, fmt, max_pairs, stream) == cudaSuccess ? IQ_OK
                                                                                                   : IQ_ERR_CUDA;
  }
  return iq::launch_gemm_rope_hadamard_fp4(tm_x, tm_w, tm_q, a, tile_n, fmt, max_pairs, stream) == cudaSuccess
             ? IQ_OK
             : IQ_ERR_CUDA;
}

bool valid_format(int fmt) { return fmt == IQ_FP4_MX || fmt == IQ_FP4_MX_OCP || fmt == IQ_FP4_NV; }

iq_status check_prepare_args(const void* latent, int M, const void* wq, const uint8_t* wq_sf, const int32_t* pos,
                             uint8_t* q_fp4, uint8_t* q_sf, const float* q_pre, bool need_pre, int fmt = IQ_FP4_MX) {
  if (M < 0 || !valid_format(fmt)) return IQ_ERR_ARG;
  if (M == 0) return IQ_OK;
  if (!latent || !wq || !wq_sf || !pos || !q_fp4 || !q_sf || (need_pre && !q_pre)) return IQ_ERR_ARG;
  if (!aligned(latent, 16) || !aligned(wq, 16) || !aligned(pos, 4) || !aligned(q_fp4, 16) ||
      !aligned(q_sf, fmt == IQ_FP4_NV ? 8 : 4) || (q_pre && !aligned(q_pre, 16))) {
    return IQ_ERR_ALIGN;
  }
  return IQ_OK;
}

iq_status prepare_impl(const void* latent, int M, const void* wq, const uint8_t* wq_sf, const int32_t* pos,
                       uint8_t* q_fp4, uint8_t* q_sf, float* q_pre, bool need_pre, void* ws, size_t ws_bytes,
                       int fmt, cudaStream_t stream) {
  iq_status st = check_prepare_args(latent, M, wq, wq_sf, pos, q_fp4, q_sf, q_pre, need_pre, fmt);
  if (st != IQ_OK || M == 0) return st;
  if (!ws) return IQ_ERR_ARG;
  if (!aligned(ws, 256)) return IQ_ERR_ALIGN;
  if (ws_bytes < iq_prepare_q_workspace(M)) return IQ_ERR_WORKSPACE;
  int max_pairs = 0;
  st = device_setup(&max_pairs);
  if (st != IQ_OK) return st;
  uint8_t* xq = static_cast<uint8_t*>(ws);
  int32_t* x_sf = reinterpret_cast<int32_t*>(xq + prepare_scales_offset(M));
  // With the fusion switched on, the CTA-pair route quantizes the token rows
  // inside the GEMM kernel (one launch); otherwise the quantizer runs first.
  if (g_quant_fusion.load(std::memory_order_relaxed) != 0 && M > g_small_m_max.load(std::memory_order_relaxed) &&
      g_tile_n_override.load(std::memory_order_relaxed) != 128) {
    const FusedQuant fuse{latent, reinterpret_cast<unsigned long long*>(xq + prepare_counters_offset(M))};
    return gemm_stage(xq, x_sf, M, wq, wq_sf, pos, q_fp4, q_sf, q_pre, fmt, max_pairs, stream, &fuse);
  }
  if (iq::launch_quant_1x128(latent, M, iq::kLatentDim, iq::kLatentDim, xq, iq::kLatentDim, x_sf, stream) !=
      cudaSuccess) {
    return IQ_ERR_CUDA;
  }
  return gemm_stage(xq, x_sf, M, wq, wq_sf, pos, q_fp4, q_sf, q_pre, fmt, max_pairs, stream);
}

}  // namespace

extern "C" {

const char* iq_status_str(iq_status s) {
  switch (s) {
    case IQ_OK: return "IQ_OK";
    case IQ_ERR_ARG: return "IQ_ERR_ARG: null pointer or invalid size";
    case IQ_ERR_ALIGN: return "IQ_ERR_ALIGN: pointer or leading dimension not aligned";
    case IQ_ERR_SHAPE: return "IQ_ERR_SHAPE: K must be positive and a multiple of 128";
    case IQ_ERR_ARCH: return "IQ_ERR_ARCH: device is not sm_103 (GB300)";
    case IQ_ERR_CUDA: return "IQ_ERR_CUDA: CUDA runtime or launch failure";
    case IQ_ERR_WORKSPACE: return "IQ_ERR_WORKSPACE: workspace too small";
    case IQ_ERR_TIMEOUT: return "IQ_ERR_TIMEOUT: a device-side wait gave up";
  }
  return "unknown iq_status";
}

iq_status iq_device_status(uint32_t* flags, int reset) {
  uint32_t v = 0, w = 0, x = 0;
  if (iq::read_device_status(&v, reset != 0) != cudaSuccess || iq::read_small_m_status(&w, reset != 0) != cudaSuccess ||
      iq::read_indexer_status(&x, reset != 0) != cudaSuccess)
    return IQ_ERR_CUDA;
  v |= w | x;
  if (flags) *flags = v;
  return v ? IQ_ERR_TIMEOUT : IQ_OK;
}

void iq_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : kDefaultTimeoutNs); }

void iq_debug_fail_next_setups(int count) { g_fail_setups.store(count > 0 ? count : 0); }

iq_status iq_debug_e2m1_codes(const float* x, long long n, uint8_t* codes, cudaStream_t stream) {
  if (n < 0) return IQ_ERR_ARG;
  if (n % 8 != 0) return IQ_ERR_SHAPE;
  if (n == 0) return IQ_OK;
  if (!x || !codes) return IQ_ERR_ARG;
  if (!aligned(x, 16) || !aligned(codes, 8)) return IQ_ERR_ALIGN;
  int max_pairs = 0;
  const iq_status st = device_setup(&max_pairs);
  if (st != IQ_OK) return st;
  return iq::launch_e2m1_codes(x, n, codes, stream) == cudaSuccess ? IQ_OK : IQ_ERR_CUDA;
}

size_t iq_selftest_workspace(void) {
  // x_sf [3][256] words, positions [256], w_sf [64][12] bytes, q_sf [256][256]
  // bytes, q_fp4 [256][4096] bytes, each at a 256-byte boundary.
  return align_up(3 * 256 * 4, 256) + align_up(256 * 4, 256) + align_up(64 * 12, 256) + 256 * 256 +
         static_cast<size_t>(256) * 4096;
}

iq_status iq_selftest_wait_timeout(void* workspace, size_t ws_bytes, uint64_t timeout_ns, uint32_t* flags,
                                   cudaStream_t stream) {
  if (!workspace || timeout_ns == 0) return IQ_ERR_ARG;
  if (!aligned(workspace, 256)) return IQ_ERR_ALIGN;
  if (ws_bytes < iq_selftest_workspace()) return IQ_ERR_WORKSPACE;
  int max_pairs = 0;
  iq_status st = device_setup(&max_pairs);
  if (st != IQ_OK) return st;
  // Start from a clean status word, so the bits read afterwards are this
  // launch's alone.
  if (cudaStreamSynchronize(stream) != cudaSuccess || iq_device_status(nullptr, 1) == IQ_ERR_CUDA) return IQ_ERR_CUDA;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  int32_t* x_sf = reinterpret_cast<int32_t*>(base);
  int32_t* pos = reinterpret_cast<int32_t*>(base + align_up(3 * 256 * 4, 256));
  uint8_t* w_sf = reinterpret_cast<uint8_t*>(pos) + align_up(256 * 4, 256);
  uint8_t* q_sf = w_sf + align_up(64 * 12, 256);
  uint8_t* q_fp4 = q_sf + 256 * 256;
  if (cudaMemsetAsync(workspace, 0, iq_selftest_workspace(), stream) != cudaSuccess) return IQ_ERR_CUDA;
  const int M = 256;
  static const iq::RopeTurns rope = make_rope_turns();
  iq::GemmArgs a{};
  a.x_sf = x_sf;
  a.w_sf = w_sf;
  a.pos = pos;
  a.q_fp4 = q_fp4;
  a.q_sf = q_sf;
  a.q_pre = nullptr;
  a.M = M;
  a.m_al = M;
  a.num_m_tiles = M / 128;
  a.num_m_pairs = 1;
  a.num_pair_tiles = iq::kQDim / 256;
  a.order = iq::kOrderFeatureMajor;
  a.timeout_ns = timeout_ns;
  a.rope = rope;
  // The tensor maps are valid descriptors over the workspace (nothing is
  // loaded through them; the store map is never used either).
  CUtensorMap tm_x, tm_w, tm_q;
  if (!encode_2d_u8(&tm_x, q_fp4, iq::kLatentDim, 256, 128, 128) ||
      !encode_2d_u8(&tm_w, q_fp4, iq::kLatentDim, 256, 128, 128) ||
      !encode_2d_u8(&tm_q, q_fp4, iq::kQDim / 2, 256, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B)) {
    return IQ_ERR_CUDA;
  }
  if (iq::launch_gemm_wait_selftest(tm_x, tm_w, tm_q, a, max_pairs, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess) {
    return IQ_ERR_CUDA;
  }
  uint32_t v = 0;
  st = iq_device_status(&v, 1);
  if (flags) *flags = v;
  return st;
}

int iq_set_small_m_threshold(int max_tokens) {
  const int v = max_tokens < 0 ? 0 : (max_tokens > iq::kSmallMMax ? iq::kSmallMMax : max_tokens);
  return g_small_m_max.exchange(v);
}

int iq_small_m_threshold(void) { return g_small_m_max.load(); }

void iq_set_gemm_tiling(int tile_n, int order) {
  g_tile_n_override.store(tile_n == 128 || tile_n == 256 ? tile_n : 0);
  g_order_override.store(order >= 1 && order <= 3 ? order : 0);
}

size_t iq_fp8_scale_words(int M, int K) {
  if (M <= 0 || K <= 0) return 0;
  return static_cast<size_t>((K + 511) / 512) * align_up(static_cast<size_t>(M), 4);
}

iq_status iq_fp8_quant_1x128_ue8m0(const void* x_bf16, int M, int K, int ldx, void* y_e4m3, int ldy,
                                   int32_t* scales, cudaStream_t stream) {
  if (M < 0) return IQ_ERR_ARG;
  if (K <= 0 || K % 128 != 0) return IQ_ERR_SHAPE;
  if (M == 0) return IQ_OK;
  if (!x_bf16 || !y_e4m3 || !scales) return IQ_ERR_ARG;
  if (ldx < K || ldy < K) return IQ_ERR_ARG;
  if (!aligned(x_bf16, 16) || !aligned(y_e4m3, 16) || !aligned(scales, 4) || ldx % 8 != 0 || ldy % 16 != 0) {
    return IQ_ERR_ALIGN;
  }
  int max_pairs = 0;
  const iq_status st = device_setup(&max_pairs);
  if (st != IQ_OK) return st;
  return iq::launch_quant_1x128(x_bf16, M, K, ldx, y_e4m3, ldy, scales, stream) == cudaSuccess ? IQ_OK
                                                                                                : IQ_ERR_CUDA;
}

size_t iq_prepare_q_workspace(int M) {
  if (M <= 0) return 0;
  return prepare_counters_offset(M) + (1 + static_cast<size_t>(iq::kMaxFusedCtas)) * sizeof(unsigned long long);
}

int iq_set_quant_fusion(int on) { return g_quant_fusion.exchange(on != 0 ? 1 : 0); }

void iq_debug_delay_quant_ns(uint64_t ns) { g_quant_delay_ns.store(ns > kMaxQuantDelayNs ? kMaxQuantDelayNs : ns); }

iq_status iq_prepare_q(const void* latent_bf16, int M, const void* wq_e4m3, const uint8_t* wq_sf,
                       const int32_t* positions, uint8_t* q_fp4, uint8_t* q_sf, void* workspace, size_t ws_bytes,
                       cudaStream_t stream) {
  return prepare_impl(latent_bf16, M, wq_e4m3, wq_sf, positions, q_fp4, q_sf, nullptr, false, workspace, ws_bytes,
                      IQ_FP4_MX, stream);
}

iq_status iq_prepare_q_debug(const void* latent_bf16, int M, const void* wq_e4m3, const uint8_t* wq_sf,
                             const int32_t* positions, uint8_t* q_fp4, uint8_t* q_sf, float* q_prequant,
                             void* workspace, size_t ws_bytes, cudaStream_t stream) {
  return prepare_impl(latent_bf16, M, wq_e4m3, wq_sf, positions, q_fp4, q_sf, q_prequant, true, workspace, ws_bytes,
                      IQ_FP4_MX, stream);
}

size_t iq_fp4_scale_bytes(int fp4_format) {
  switch (fp4_format) {
    case IQ_FP4_MX:
    case IQ_FP4_MX_OCP: return iq::Fp4Layout<iq::kFp4Mx>::kScaleBytesPerToken;
    case IQ_FP4_NV: return iq::Fp4Layout<iq::kFp4Nv>::kScaleBytesPerToken;
  }
  return 0;
}

iq_status iq_prepare_q_ex(const void* latent_bf16, int M, const void* wq_e4m3, const uint8_t* wq_sf,
                          const int32_t* positions, int fp4_format, uint8_t* q_fp4, uint8_t* q_sf, float* q_prequant,
                          void* workspace, size_t ws_bytes, cudaStream_t stream) {
  return prepare_impl(latent_bf16, M, wq_e4m3, wq_sf, positions, q_fp4, q_sf, q_prequant, false, workspace, ws_bytes,
                      fp4_format, stream);
}

iq_status iq_gemm_rope_hadamard_fp4(const void* xq_e4m3, const int32_t* x_scales, int M, const void* wq_e4m3,
                                    const uint8_t* wq_sf, const int32_t* positions, uint8_t* q_fp4, uint8_t* q_sf,
                                    float* q_prequant, cudaStream_t stream) {
  iq_status st = check_prepare_args(xq_e4m3, M, wq_e4m3, wq_sf, positions, q_fp4, q_sf, q_prequant, false);
  if (st != IQ_OK || M == 0) return st;
  if (!x_scales) return IQ_ERR_ARG;
  if (!aligned(x_scales, 4)) return IQ_ERR_ALIGN;
  int max_pairs = 0;
  st = device_setup(&max_pairs);
  if (st != IQ_OK) return st;
  return gemm_stage(xq_e4m3, x_scales, M, wq_e4m3, wq_sf, positions, q_fp4, q_sf, q_prequant, IQ_FP4_MX, max_pairs,
                    stream);
}

}  // extern "C"

// ------------------------------------------------------------------------
// iq_prepare_q_static: the indexer-Q preparation for callers that cannot
// allocate device memory.  The FP8 latent and its scale words go to a scratch
// array compiled into the library instead of a caller workspace.

namespace {

constexpr size_t kStaticLatentBytes = static_cast<size_t>(IQ_STATIC_MAX_TOKENS) * iq::kLatentDim;
constexpr size_t kStaticScratchBytes =
    (kStaticLatentBytes + 255) / 256 * 256 + static_cast<size_t>(iq::kScaleGroups) * IQ_STATIC_MAX_TOKENS * 4;

// One scratch array per device, alive until the process exits.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mutex;
void* g_static_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name stands for a host-side shadow, not device memory, so the
// address is looked up once per device (with that device current) and cached.
iq_status static_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return IQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (g_static_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return IQ_ERR_CUDA;
    g_static_scratch_addr[dev] = p;
  }
  *out = g_static_scratch_addr[dev];
  return IQ_OK;
}

}  // namespace

extern "C" iq_status iq_prepare_q_static(const void* latent_bf16, int M, const void* wq_e4m3, const uint8_t* wq_sf,
                                         const int32_t* positions, uint8_t* q_fp4, uint8_t* q_sf,
                                         cudaStream_t stream) {
  iq_status st = check_prepare_args(latent_bf16, M, wq_e4m3, wq_sf, positions, q_fp4, q_sf, nullptr, false);
  if (st != IQ_OK || M == 0) return st;
  if (M > IQ_STATIC_MAX_TOKENS) return IQ_ERR_WORKSPACE;
  int max_pairs = 0;
  st = device_setup(&max_pairs);
  if (st != IQ_OK) return st;
  void* scratch = nullptr;
  st = static_scratch_address(&scratch);
  if (st != IQ_OK) return st;
  uint8_t* xq = static_cast<uint8_t*>(scratch);
  int32_t* x_sf = reinterpret_cast<int32_t*>(xq + align_up(static_cast<size_t>(M) * iq::kLatentDim, 256));
  if (iq::launch_quant_1x128(latent_bf16, M, iq::kLatentDim, iq::kLatentDim, xq, iq::kLatentDim, x_sf, stream) !=
      cudaSuccess) {
    return IQ_ERR_CUDA;
  }
  return gemm_stage(xq, x_sf, M, wq_e4m3, wq_sf, positions, q_fp4, q_sf, nullptr, IQ_FP4_MX, max_pairs, stream);
}

// ---------------------------------------------------------------------------
// Host-buffer entry: row chunks pipelined over the host link.  Three internal
// streams per device: `in` runs the quantizer of chunk c, which reads the
// chunk's latent rows and positions straight from page-locked host memory;
// `comp` (highest priority) runs the GEMM of chunk c once its quantizer is
// done; `out` copies chunk c's FP4 codes and scales to the host once its GEMM
// is done.  Chunk c + 1's quantizer therefore runs beside chunk c's GEMM (one
// block per SM next to the GEMM's CTA) while chunk c - 1's results travel
// back, and the link carries both directions at once.

namespace {

constexpr int kHostChunkAlign = 256;      // chunk starts stay on CTA-pair tile boundaries
constexpr int kMaxHostChunks = 64;
constexpr int kDefaultHostChunkRows = 1024;
std::atomic<int> g_host_chunk_rows{kDefaultHostChunkRows};

struct HostPath {
  std::mutex mu;                          // one call at a time enqueues on the internal streams
  bool ready = false;
  iq_status status = IQ_OK;
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t fork = nullptr, tail_in = nullptr, tail_comp = nullptr, join = nullptr;
  cudaEvent_t in_done[kMaxHostChunks] = {};
  cudaEvent_t comp_done[kMaxHostChunks] = {};
};
HostPath g_host[kMaxDevices];

// Streams and events of the host-buffer entry on the current device, created
// by its first call there (with the device's lock held).
iq_status host_path_setup(HostPath& h) {
  if (h.ready) return h.status;
  h.ready = true;
  int least = 0, greatest = 0;
  const unsigned ev = cudaEventDisableTiming;
  bool ok = cudaDeviceGetStreamPriorityRange(&least, &greatest) == cudaSuccess &&
            cudaStreamCreateWithPriority(&h.comp, cudaStreamNonBlocking, greatest) == cudaSuccess &&
            cudaStreamCreateWithPriority(&h.in, cudaStreamNonBlocking, least) == cudaSuccess &&
            cudaStreamCreateWithPriority(&h.out, cudaStreamNonBlocking, least) == cudaSuccess &&
            cudaEventCreateWithFlags(&h.fork, ev) == cudaSuccess &&
            cudaEventCreateWithFlags(&h.tail_in, ev) == cudaSuccess &&
            cudaEventCreateWithFlags(&h.tail_comp, ev) == cudaSuccess &&
            cudaEventCreateWithFlags(&h.join, ev) == cudaSuccess;
  for (int i = 0; ok && i < kMaxHostChunks; ++i) {
    ok = cudaEventCreateWithFlags(&h.in_done[i], ev) == cudaSuccess &&
         cudaEventCreateWithFlags(&h.comp_done[i], ev) == cudaSuccess;
  }
  h.status = ok ? IQ_OK : IQ_ERR_CUDA;
  return h.status;
}

// The address at which kernels on device `dev` reach a caller buffer that is
// page-locked host memory, or device / managed memory of that device; nullptr
// for pageable host memory or another device's memory.
const void* device_view(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  switch (a.type) {
    case cudaMemoryTypeHost:
      return a.devicePointer;
    case cudaMemoryTypeDevice:
      return a.device == dev ? p : nullptr;
    case cudaMemoryTypeManaged:
      return p;
    default:
      return nullptr;
  }
}

// Device workspace of the host-buffer entry: FP4 codes, FP4 scales and
// positions of all M rows, then the FP8 latent and its packed scales.  Chunk
// starts are multiples of 256 rows, so every chunk's packed-scale array
// (3 groups x align4(rows) words) starts 3 * (first row) words in.
size_t host_ws_bytes(int M, size_t sfb) {
  const size_t m = static_cast<size_t>(M);
  return align_up(m * (iq::kQDim / 2), 256) + align_up(m * sfb, 256) + align_up(m * sizeof(int32_t), 256) +
         align_up(m * iq::kLatentDim, 256) + iq::kScaleGroups * align_up(m, 4) * sizeof(int32_t);
}

}  // namespace

extern "C" size_t iq_prepare_q_host_workspace(int M, int fp4_format) {
  if (M <= 0 || !valid_format(fp4_format)) return 0;
  return host_ws_bytes(M, iq_fp4_scale_bytes(fp4_format));
}

extern "C" int iq_set_host_chunk_rows(int rows) {
  if (rows < kHostChunkAlign) rows = kHostChunkAlign;
  if (rows > (1 << 20)) rows = 1 << 20;
  rows = (rows + kHostChunkAlign - 1) / kHostChunkAlign * kHostChunkAlign;
  return g_host_chunk_rows.exchange(rows);
}

extern "C" int iq_host_chunk_rows(void) { return g_host_chunk_rows.load(); }

extern "C" iq_status iq_prepare_q_host(const void* latent_bf16, int M, const void* wq_e4m3, const uint8_t* wq_sf,
                                       const int32_t* positions, int fp4_format, uint8_t* q_fp4, uint8_t* q_sf,
                                       void* workspace, size_t ws_bytes, cudaStream_t stream) {
  iq_status st =
      check_prepare_args(latent_bf16, M, wq_e4m3, wq_sf, positions, q_fp4, q_sf, nullptr, false, fp4_format);
  if (st != IQ_OK || M == 0) return st;
  if (!workspace) return IQ_ERR_ARG;
  if (!aligned(workspace, 256)) return IQ_ERR_ALIGN;
  const size_t sfb = iq_fp4_scale_bytes(fp4_format);
  if (ws_bytes < host_ws_bytes(M, sfb)) return IQ_ERR_WORKSPACE;
  int max_pairs = 0, sm_count = 0;
  st = device_setup(&max_pairs, &sm_count);
  if (st != IQ_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IQ_ERR_CUDA;
  const uint16_t* lat = static_cast<const uint16_t*>(device_view(latent_bf16, dev));
  const int32_t* pos_src = static_cast<const int32_t*>(device_view(positions, dev));
  if (!lat || !pos_src || !device_view(q_fp4, dev) || !device_view(q_sf, dev)) return IQ_ERR_ARG;

  HostPath& h = g_host[dev];
  std::lock_guard<std::mutex> lock(h.mu);
  st = host_path_setup(h);
  if (st != IQ_OK) return st;

  const size_t m = static_cast<size_t>(M);
  uint8_t* q_dev = static_cast<uint8_t*>(workspace);
  uint8_t* sf_dev = q_dev + align_up(m * (iq::kQDim / 2), 256);
  int32_t* pos_dev = reinterpret_cast<int32_t*>(sf_dev + align_up(m * sfb, 256));
  uint8_t* xq = reinterpret_cast<uint8_t*>(pos_dev) + align_up(m * sizeof(int32_t), 256);
  int32_t* x_sf = reinterpret_cast<int32_t*>(xq + align_up(m * iq::kLatentDim, 256));

  int rows = g_host_chunk_rows.load(std::memory_order_relaxed);
  const int min_rows = (M + kMaxHostChunks - 1) / kMaxHostChunks;
  if (rows < min_rows) rows = (min_rows + kHostChunkAlign - 1) / kHostChunkAlign * kHostChunkAlign;
  const int chunks = (M + rows - 1) / rows;

  bool ok = cudaEventRecord(h.fork, stream) == cudaSuccess && cudaStreamWaitEvent(h.in, h.fork, 0) == cudaSuccess &&
            cudaStreamWaitEvent(h.comp, h.fork, 0) == cudaSuccess &&
            cudaStreamWaitEvent(h.out, h.fork, 0) == cudaSuccess;
  for (int c = 0; ok && c < chunks; ++c) {
    const int r0 = c * rows;
    const int mc = M - r0 < rows ? M - r0 : rows;
    const size_t q_off = static_cast<size_t>(r0) * (iq::kQDim / 2), sf_off = static_cast<size_t>(r0) * sfb;
    uint8_t* xq_c = xq + static_cast<size_t>(r0) * iq::kLatentDim;
    int32_t* x_sf_c = x_sf + static_cast<size_t>(iq::kScaleGroups) * r0;
    ok = iq::launch_quant_1x128_host_rows(lat + static_cast<size_t>(r0) * iq::kLatentDim, mc, iq::kLatentDim,
                                          iq::kLatentDim, xq_c, iq::kLatentDim, x_sf_c, pos_src + r0, pos_dev + r0,
                                          sm_count, h.in) == cudaSuccess &&
         cudaEventRecord(h.in_done[c], h.in) == cudaSuccess &&
         cudaStreamWaitEvent(h.comp, h.in_done[c], 0) == cudaSuccess;
    if (ok) {
      // The GEMM kernels are launched with programmatic stream serialization
      // but never trigger an early launch themselves, so a chunk's GEMM starts
      // after the previous chunk's has completed, and after the event wait
      // above (its inputs come from another stream).
      st = gemm_stage(xq_c, x_sf_c, mc, wq_e4m3, wq_sf, pos_dev + r0, q_dev + q_off, sf_dev + sf_off, nullptr,
                      fp4_format, max_pairs, h.comp);
      ok = st == IQ_OK;
    }
    ok = ok && cudaEventRecord(h.comp_done[c], h.comp) == cudaSuccess &&
         cudaStreamWaitEvent(h.out, h.comp_done[c], 0) == cudaSuccess &&
         cudaMemcpyAsync(q_fp4 + q_off, q_dev + q_off, static_cast<size_t>(mc) * (iq::kQDim / 2), cudaMemcpyDefault,
                         h.out) == cudaSuccess &&
         cudaMemcpyAsync(q_sf + sf_off, sf_dev + sf_off, static_cast<size_t>(mc) * sfb, cudaMemcpyDefault, h.out) ==
             cudaSuccess;
  }
  // Join all three streams back into `stream`, also after a failed step, so
  // that later work on `stream` stays ordered after everything enqueued here.
  const bool joined = cudaEventRecord(h.tail_in, h.in) == cudaSuccess &&
                      cudaEventRecord(h.tail_comp, h.comp) == cudaSuccess &&
                      cudaStreamWaitEvent(h.out, h.tail_in, 0) == cudaSuccess &&
                      cudaStreamWaitEvent(h.out, h.tail_comp, 0) == cudaSuccess &&
                      cudaEventRecord(h.join, h.out) == cudaSuccess &&
                      cudaStreamWaitEvent(stream, h.join, 0) == cudaSuccess;
  if (st != IQ_OK) return st;
  return ok && joined ? IQ_OK : IQ_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Downstream indexer: scores and top-k selection.

extern "C" iq_status iq_indexer_logits(const uint8_t* q_fp4, const uint8_t* q_sf, int M, const uint8_t* k_fp4,
                                       const uint8_t* k_sf, int N, const float* weights, const int32_t* lengths,
                                       float* logits, long long ld_logits, cudaStream_t stream) {
  if (M < 0 || N < 0) return IQ_ERR_ARG;
  if (M == 0 || N == 0) return IQ_OK;
  if (!q_fp4 || !q_sf || !k_fp4 || !k_sf || !weights || !lengths || !logits || ld_logits < N) return IQ_ERR_ARG;
  if (!aligned(q_fp4, 16) || !aligned(k_fp4, 16) || !aligned(q_sf, 16) || !aligned(k_sf, 16) || !aligned(weights, 16) ||
      !aligned(lengths, 4) || !aligned(logits, 4)) {
    return IQ_ERR_ALIGN;
  }
  if (static_cast<long long>(M) * iq::kNumHeads > (1ll << 31) - 1) return IQ_ERR_ARG;
  int max_pairs = 0, sm_count = 0;
  const iq_status st = device_setup(&max_pairs, &sm_count);
  if (st != IQ_OK) return st;
  CUtensorMap tm_k, tm_q;
  if (!encode_2d_u8(&tm_k, k_fp4, iq::kHeadDim / 2, static_cast<uint64_t>(N), 64, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !encode_2d_u8(&tm_q, q_fp4, iq::kHeadDim / 2, static_cast<uint64_t>(M) * iq::kNumHeads, 64, 256,
                    CU_TENSOR_MAP_SWIZZLE_64B)) {
    return IQ_ERR_CUDA;
  }
  return iq::launch_indexer_logits(tm_k, tm_q, q_sf, k_sf, weights, lengths, logits, ld_logits, M, N, sm_count,
                                   g_timeout_ns.load(std::memory_order_relaxed), stream) == cudaSuccess
             ? IQ_OK
             : IQ_ERR_CUDA;
}

extern "C" iq_status iq_indexer_topk(const float* logits, long long ld_logits, int M, int N, const int32_t* lengths,
                                     int k, int32_t* indices, cudaStream_t stream) {
  if (M < 0 || N < 0 || k < 1) return IQ_ERR_ARG;
  if (M == 0) return IQ_OK;
  if (!logits || !lengths || !indices || ld_logits < N) return IQ_ERR_ARG;
  if (!aligned(logits, 4) || !aligned(lengths, 4) || !aligned(indices, 4)) return IQ_ERR_ALIGN;
  int max_pairs = 0;
  const iq_status st = device_setup(&max_pairs);
  if (st != IQ_OK) return st;
  return iq::launch_indexer_topk(logits, ld_logits, M, N, lengths, k, indices, stream) == cudaSuccess ? IQ_OK
                                                                                                      : IQ_ERR_CUDA;
}
