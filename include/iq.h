/*
 * iq.h -- C ABI of the GB300 (sm_103a) DeepSeek-V4 indexer-Q preparation path.
 *
 * Two operations, each an asynchronous launch sequence on a caller stream:
 *
 *  1. iq_fp8_quant_1x128_ue8m0: the packed-UE8M0 FP8 online activation
 *     quantizer of the TokenSpeed PR "perf(deepseek-v4): accelerate indexer Q
 *     and packed FP8 quantization" (Summary; Risk and fallback: contiguous,
 *     aligned BF16 input, K divisible by 128, the packed-UE8M0 scale contract
 *     and the tiny-scale floor), which the TensorRT-LLM PR "Fuse DeepSeek-V4
 *     Indexer Q projection with CuTe DSL" calls fp8_quantize_1x128 with UE8M0
 *     scales (Walkthrough / sequence diagram).
 *
 *  2. iq_prepare_q: the fused indexer-Q projection of the TensorRT-LLM PR
 *     (sequence diagram: FP8 input and UE8M0 scales, block-scaled GEMM "with
 *     RoPE and FP4 epilogue", packed FP4 Q and scales returned; review comment
 *     on the fused epilogue: MXF8 scale vector 32, one 128-column head per MMA
 *     tile) with the Hadamard transform that the TokenSpeed PR applies to the
 *     indexer Q (Summary; Main-rebase compatibility fix).
 *
 * Numbers used throughout (element formats per the OCP FP8 / MX specs):
 *   E4M3: FP8 with 4 exponent bits (bias 7), 3 mantissa bits, max 448.
 *   E2M1: FP4 with 2 exponent bits (bias 1), 1 mantissa bit, max 6.
 *   UE8M0: unsigned 8-bit exponent; byte b encodes 2^(b - 127).
 *   Block scale exponent of a block with largest magnitude a:
 *       e = smallest integer with qmax * 2^e >= max(a, 1e-4)   (qmax 448 or 6)
 *   Element code = round-to-nearest-even(x * 2^-e) in the element format.
 *
 * Memory: the caller owns every buffer (inputs, outputs, workspace).  No call
 * allocates device memory or falls back to another implementation, and none
 * synchronizes the device or the stream except the diagnostics
 * (iq_device_status, iq_selftest_wait_timeout).  Pointers are device pointers unless stated.
 * All calls are asynchronous on `stream`; errors detected on the host are
 * returned before anything is launched.  A return of IQ_OK means the launches
 * were enqueued; a device-side wait that ran out of time is recorded in the
 * device status word (iq_device_status).
 *
 * Thread safety: calls may be made from several host threads.  Shared host
 * state: the per-device set-up done on the first call on a device
 * (architecture check, kernel attributes), which is guarded, and the
 * internal streams and events of iq_prepare_q_host, whose calls on one device
 * enqueue one at a time under a lock.
 */
#ifndef IQ_H_
#define IQ_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  IQ_OK = 0,
  IQ_ERR_ARG = -1,        /* null pointer, M < 0, bad leading dimension */
  IQ_ERR_ALIGN = -2,      /* a pointer or leading dimension breaks the alignment rule */
  IQ_ERR_SHAPE = -3,      /* K <= 0 or K % 128 != 0 */
  IQ_ERR_ARCH = -4,       /* current device is not compute capability 10.3 (sm_103) */
  IQ_ERR_CUDA = -5,       /* a CUDA runtime call or launch failed */
  IQ_ERR_WORKSPACE = -6,  /* workspace smaller than iq_prepare_q_workspace(M) */
  IQ_ERR_TIMEOUT = -7     /* a device-side wait gave up (see iq_device_status) */
} iq_status;

/* Human-readable name of a status code (static storage). */
const char* iq_status_str(iq_status s);

/* Device-side status word of the current device: bit i set means a wait of
 * kind i ran out of time in some launch since the last reset.  Reads it into
 * *flags (may be NULL) and clears it when `reset` is nonzero.  This call
 * synchronizes with the device (it copies from device memory); it is a
 * diagnostic, not part of the hot path.  Returns IQ_ERR_TIMEOUT when the word
 * was nonzero, IQ_OK otherwise. */
iq_status iq_device_status(uint32_t* flags, int reset);

/* Overrides the time after which a device-side wait gives up, in nanoseconds
 * (default 2e9).  0 restores the default.  Applies to later launches from any
 * thread. */
void iq_set_wait_timeout_ns(uint64_t ns);

/* Diagnostics of the failure handling (no counterpart on the pages).
 *
 * iq_selftest_wait_timeout runs the fused GEMM kernel once on a 256-token
 * problem with its TMA loads left out: the stage barriers its MMA issuer
 * waits on never complete, no MMA is issued, and the producer's, the MMA
 * issuer's and the epilogue's bounded waits give up after timeout_ns with
 * nothing asynchronous in flight.  The kernel then takes its normal give-up
 * and teardown path.  The call resets the status word, launches on `stream`,
 * synchronizes the stream, stores the status bits the launch set in *flags
 * (may be NULL) and resets the word again.  Returns IQ_ERR_TIMEOUT when some
 * wait gave up (the expected result: bits 0, 1 and 2 -- producer, MMA issuer,
 * epilogue -- set, bit 3 -- teardown -- clear), IQ_OK when none did.
 * workspace: iq_selftest_workspace() bytes of device memory, 256-byte
 * aligned, overwritten.  Errors: IQ_ERR_ARG (NULL workspace, timeout 0),
 * IQ_ERR_ALIGN, IQ_ERR_WORKSPACE, IQ_ERR_CUDA, IQ_ERR_ARCH. */
size_t iq_selftest_workspace(void);
iq_status iq_selftest_wait_timeout(void* workspace, size_t ws_bytes, uint64_t timeout_ns, uint32_t* flags,
                                   cudaStream_t stream);

/* Test hook: the next `count` per-device set-ups (the work of the first call
 * on a device) fail as if a CUDA query had failed and return IQ_ERR_CUDA.  A
 * failed set-up is not cached: the next call on the device tries again. */
void iq_debug_fail_next_setups(int count);

/* The FP4 stage's element conversion alone, for testing it directly:
 * codes[i] (low nibble) = E2M1 code of x[i], round to nearest even,
 * saturating at +-6, sign of zero kept -- the conversion both fused GEMM
 * kernels apply to z * 2^-e.  x: n float32, 16-byte aligned; codes: n bytes,
 * 8-byte aligned; n % 8 == 0 (else IQ_ERR_SHAPE).  One kernel launch. */
iq_status iq_debug_e2m1_codes(const float* x, long long n, uint8_t* codes, cudaStream_t stream);

/* Token-count route of the fused GEMM (operation 2).  Calls with
 * 1 <= M <= threshold run the small-M kernel, which swaps the MMA operands
 * (the weights on the MMA's M side, the tokens on its N side: 64 token
 * columns up to 64 tokens, 128 above), the variant the TensorRT-LLM PR routes
 * small token counts to (dispatch thresholds); larger M runs the persistent
 * CTA-pair kernel.  Both compute the same operation;
 * their float32 sums may round differently, within the error the parity rules
 * of operation 2 allow.  The threshold is clamped to [0, IQ_SMALL_M_MAX]; 0
 * sends every M to the CTA-pair kernel.  The default is IQ_SMALL_M_MAX.
 * Process-wide; applies to later calls from any thread (a CUDA graph keeps
 * the route it was captured with).  Returns the previous threshold. */
#define IQ_SMALL_M_MAX 128
int iq_set_small_m_threshold(int max_tokens);

/* The current threshold (see iq_set_small_m_threshold). */
int iq_small_m_threshold(void);

/* Tuning override of the CTA-pair kernel's tiling, for measurements.  By
 * default the kernel takes one head (128 output features) per pair tile up to
 * 256 tokens and two heads (256) above, and orders the pair tiles token-major
 * (consecutive tiles of a CTA pair share their 256 token rows).  tile_n: 128 (one head per tile, two accumulators
 * in tensor memory) or 256 forces that width, any other value restores the
 * default; order: 1 forces feature-major (consecutive tiles share their
 * heads), 2 token-major, 3 interleaved (token-major tiles dealt round-robin
 * to the pairs: pair p takes tiles p, p + P, ...), any other value restores
 * the default.
 * Results are the same under every setting (the same sums in the same order
 * per output).  Process-wide; applies to later calls. */
void iq_set_gemm_tiling(int tile_n, int order);

/* The quantizer fused into the CTA-pair kernel: off (0, the default: the
 * stand-alone quantizer, then the GEMM kernel) or on (1: one launch, see
 * iq_prepare_q).  Results are the same either way; on GB300 the fused launch
 * measured slower at every token count, so it is off unless asked for.  The
 * fused launch always takes two-head tiles; forcing one-head tiles
 * (iq_set_gemm_tiling) turns it off.  Process-wide; applies to later calls;
 * returns the previous setting. */
int iq_set_quant_fusion(int on);

/* Diagnostics: the fused quantizer's warps wait ns nanoseconds (at most 1 ms)
 * before signalling each wave of token rows, so that the GEMM's loads must
 * wait for them.  0 (the default) turns it off.  Process-wide. */
void iq_debug_delay_quant_ns(uint64_t ns);

/* ------------------------------------------------------------------------
 * 1. FP8 1x128 quantizer with packed UE8M0 scales.
 * ------------------------------------------------------------------------ */

/* Number of int32 scale words the quantizer writes for an M x K input:
 * ceil(K / 512) * align_up(M, 4).  Returns 0 when M <= 0 or K <= 0. */
size_t iq_fp8_scale_words(int M, int K);

/* Quantizes x (BF16, row-major [M, ldx], first K columns used) per row and
 * per 1x128 block:
 *   y[m, k]   = E4M3 code of x[m, k] * 2^-e(m, k/128)        (row-major [M, ldy])
 *   scales    = int32 words [ceil(K/512)][align_up(M, 4)] (M-major, the
 *               TMA-aligned layout a DeepGEMM-style consumer reads):
 *               byte j (little-endian) of word [g][m] is the UE8M0 scale byte
 *               e + 127 of block 4g + j of row m; bytes of blocks past K/128
 *               and words of rows m >= M are written as 0.
 * The sign of zero is kept (-0 and values that round to zero from below give
 * code 0x80).  NaN or infinite inputs are outside the contract.
 * Requirements: M >= 0; K > 0 and K % 128 == 0 (else IQ_ERR_SHAPE);
 *   ldx >= K, ldy >= K; x and y 16-byte aligned, ldx % 8 == 0 and
 *   ldy % 16 == 0, scales 4-byte aligned (else IQ_ERR_ALIGN).
 * M == 0 returns IQ_OK without a launch.  One kernel launch, with programmatic
 * stream serialization: its blocks may be scheduled while the preceding
 * kernel on `stream` runs, and they touch no memory before that kernel has
 * completed. */
iq_status iq_fp8_quant_1x128_ue8m0(const void* x_bf16, int M, int K, int ldx,
                                   void* y_e4m3, int ldy, int32_t* scales,
                                   cudaStream_t stream);

/* ------------------------------------------------------------------------
 * 2. Indexer-Q preparation: FP8 quantize -> block-scaled FP8 GEMM -> RoPE ->
 *    Hadamard-128 -> FP4 (E2M1) with 1x32 UE8M0 scales.
 *
 * Fixed shapes: latent dimension K = 1536; Q has 64 heads of 128 dims
 * (N = 8192).  Per token m and head h (n = 128 h + d):
 *   Y[m, n] = sum_kb 2^(eX[m,kb] + eW[h,kb]) * sum_{k in kb} x[m,k] w[n,k]
 *             over 12 blocks kb of 128, x the E4M3 latent codes (operation 1
 *             applied to the BF16 latent), w the weight codes;
 *   RoPE:     NeoX rotation of dims d = 0..63 in pairs (i, i+32) by the angle
 *             position[m] * 10000^(-i/32); dims 64..127 unchanged;
 *   Hadamard: z = H r / sqrt(128), H[i][j] = (-1)^popcount(i & j);
 *   FP4:      per block of 32 consecutive dims, e from qmax 6, codes
 *             E2M1(z * 2^-e) with the sign of zero kept.
 * The pre-quant Q (z) is kept in float32 and is never rounded to BF16.
 * ------------------------------------------------------------------------ */

#define IQ_LATENT_DIM 1536
#define IQ_NUM_HEADS 64
#define IQ_HEAD_DIM 128
#define IQ_Q_DIM 8192

/* Workspace bytes iq_prepare_q needs for M tokens: the E4M3 latent
 * [M, 1536] at offset 0 followed, at the next 256-byte boundary, by its packed
 * scale words [3][align_up(M, 4)], then, at the next 256-byte boundary, the
 * fused quantizer's flags (513 words of 8 bytes: a call counter and one
 * progress word per CTA).  The flags need no initialisation: a progress word
 * counts only if it carries a 48-bit hash of the current call counter and its
 * CTA, which each call advances.  Returns 0 when M <= 0. */
size_t iq_prepare_q_workspace(int M);

/* Arguments:
 *   latent_bf16  [M, 1536] BF16, contiguous, 16-byte aligned.
 *   wq_e4m3      [8192, 1536] E4M3 codes, row-major (row n = output feature n),
 *                16-byte aligned.
 *   wq_sf        [64][12] UE8M0 bytes, row-major: scale of the 128x128 weight
 *                block (head h, K-block kb).
 *   positions    [M] int32 token positions (any value with |p| < 2^24).
 *   q_fp4        [M, 4096] bytes, 16-byte aligned: byte 64 h + 16 b + i of
 *                row m holds dims 32 b + 2i (low nibble) and 32 b + 2i + 1
 *                (high nibble) of head h.
 *   q_sf         [M, 256] UE8M0 bytes, 4-byte aligned: byte 4 h + b is the
 *                scale of block b of head h.
 *   workspace    caller scratch of at least iq_prepare_q_workspace(M) bytes,
 *                256-byte aligned; its contents on return are the FP8 latent
 *                and its packed scales (operation 1's outputs).
 * M == 0 returns IQ_OK without a launch.
 *
 * Launches.  Two kernel launches, back to back on `stream`: the quantizer,
 * then the GEMM kernel of M's route (see iq_set_small_m_threshold), launched
 * as the quantizer's programmatic dependent so that its set-up (and, on the
 * small-M route, its weight loads) overlap the quantizer.  With the fusion
 * switched on (iq_set_quant_fusion) the CTA-pair route is ONE launch: the
 * GEMM kernel quantizes the token rows itself (operation 1's arithmetic, the
 * same codes and scale words in the workspace) in waves ahead of the tiles
 * that read them, and a tile's loads wait for the progress flags of the CTAs
 * that quantized its rows; that launch is cooperative (all of its CTAs, one
 * per SM, resident at once).
 *
 * Ordering: the GEMM kernels of both routes read wq_e4m3 and wq_sf before the
 * kernel launched just before them on `stream` has completed (that kernel is
 * the quantizer for iq_prepare_q; for iq_gemm_rope_hadamard_fp4 it is
 * whatever the caller launched last, and the overlap happens only if that
 * kernel allows programmatic dependents).  The weights must therefore not be
 * written by the immediately preceding kernel.  Every other input is read
 * after that kernel has completed; the quantizer, itself launched as a
 * programmatic dependent of whatever precedes it, touches no memory before
 * that.  The kernels let the next kernel on `stream` be scheduled while they
 * run (griddepcontrol.launch_dependents): a following kernel launched with
 * programmatic stream serialization must wait for them
 * (griddepcontrol.wait) before it reads this call's outputs or workspace, as
 * that launch mode requires of any kernel.  Calls that run at the same time
 * must not share a workspace; calls enqueued one after another on one stream
 * may. */
iq_status iq_prepare_q(const void* latent_bf16, int M,
                       const void* wq_e4m3, const uint8_t* wq_sf,
                       const int32_t* positions,
                       uint8_t* q_fp4, uint8_t* q_sf,
                       void* workspace, size_t ws_bytes, cudaStream_t stream);

/* iq_prepare_q that also writes the float32 pre-quant Q (z above) to
 * q_prequant [M, 8192] (row-major, 16-byte aligned). */
iq_status iq_prepare_q_debug(const void* latent_bf16, int M,
                             const void* wq_e4m3, const uint8_t* wq_sf,
                             const int32_t* positions,
                             uint8_t* q_fp4, uint8_t* q_sf, float* q_prequant,
                             void* workspace, size_t ws_bytes, cudaStream_t stream);

/* The second stage alone, for callers that already hold the FP8 latent and its
 * packed scales (the outputs of operation 1 with K = 1536):
 *   xq_e4m3      [M, 1536] E4M3 codes, contiguous, 16-byte aligned.
 *   x_scales     [3][align_up(M, 4)] packed UE8M0 words, 4-byte aligned.
 *   q_prequant   may be NULL; otherwise as in iq_prepare_q_debug.
 * One kernel launch. */
iq_status iq_gemm_rope_hadamard_fp4(const void* xq_e4m3, const int32_t* x_scales, int M,
                                    const void* wq_e4m3, const uint8_t* wq_sf,
                                    const int32_t* positions,
                                    uint8_t* q_fp4, uint8_t* q_sf, float* q_prequant,
                                    cudaStream_t stream);

/* ------------------------------------------------------------------------
 * FP4 output variants.  iq_prepare_q writes MXFP4 with the scale rule above
 * (IQ_FP4_MX).  iq_prepare_q_ex selects one of:
 *   IQ_FP4_MX      1x32 blocks, UE8M0 scale 2^e, e the smallest integer with
 *                  6 * 2^e >= max(amax, 1e-4); never saturates.  q_sf [M, 256].
 *   IQ_FP4_MX_OCP  1x32 blocks, UE8M0 scale 2^e with e = floor(log2(max(amax,
 *                  1e-4))) - 2, the shared-scale rule of the OCP Microscaling
 *                  (MX) spec for E2M1; elements saturate at 6.  q_sf [M, 256].
 *   IQ_FP4_NV      1x16 blocks with an E4M3 scale s (NVFP4-style, per-tensor
 *                  scale 1): s = round-to-nearest-even E4M3 of
 *                  float32(max(amax, 1e-4) / 6), or 2^-9 (code 1) when that
 *                  rounds to zero; codes E2M1(float32(z * float32(1 / s))),
 *                  saturating at 6.  q_sf [M, 512] E4M3 bytes, byte 8 h + b the
 *                  scale of block b (dims 16 b .. 16 b + 15) of head h; 8-byte
 *                  aligned.
 * The pages specify only the MXFP4 output; the other two are variants of the
 * same FP4 stage for consumers that expect them.
 * ------------------------------------------------------------------------ */

typedef enum { IQ_FP4_MX = 0, IQ_FP4_MX_OCP = 1, IQ_FP4_NV = 2 } iq_fp4_format;

/* Scale bytes per token of a format (256 or 512); 0 for an unknown format. */
size_t iq_fp4_scale_bytes(int fp4_format);

/* iq_prepare_q with the FP4 output variant `fp4_format` (iq_fp4_format);
 * q_sf holds iq_fp4_scale_bytes(fp4_format) bytes per token; q_prequant may
 * be NULL, else it receives the float32 pre-quant Q as in iq_prepare_q_debug.
 * An unknown format returns IQ_ERR_ARG. */
iq_status iq_prepare_q_ex(const void* latent_bf16, int M,
                          const void* wq_e4m3, const uint8_t* wq_sf,
                          const int32_t* positions, int fp4_format,
                          uint8_t* q_fp4, uint8_t* q_sf, float* q_prequant,
                          void* workspace, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Indexer-Q preparation without any device allocation.  The pages have no
 * counterpart of this call; it exists for callers that cannot obtain device
 * memory at the point where they prepare Q -- for example a plugin whose host
 * program owns every device allocation and offers it no allocator, or a
 * latency-bound loop that must not call cudaMalloc (which can synchronize the
 * device).  Such a caller passes only inputs and outputs.
 *
 * The FP8 latent and its packed scales, which iq_prepare_q keeps in the
 * caller's workspace, live instead in one scratch array built into the
 * library: IQ_STATIC_MAX_TOKENS * 1536 bytes plus the scale words (about
 * 3.2 MB), held on every GPU that loads the library until the process exits.
 *
 * Behaviour:
 *  - M > IQ_STATIC_MAX_TOKENS returns IQ_ERR_WORKSPACE (the built-in scratch
 *    is too small) before anything is launched; M == 0 returns IQ_OK.
 *  - The first call on a device looks up the device address of the scratch
 *    array (cudaGetSymbolAddress) with that device current; make that first
 *    call before any stream capture on the device.
 *  - All calls on a device share the one scratch array, and it keeps what the
 *    previous call left there.  Nothing in it needs clearing: every byte the
 *    GEMM kernel reads is written by the quantizer kernel of the same call.
 *    Calls whose work overlaps on the GPU (for example on two streams without
 *    ordering between them) race on the scratch and give wrong results;
 *    order them on one stream or with events.
 *  - Same arguments, results and errors as iq_prepare_q otherwise; nothing
 *    is allocated, no allocating library routine is called.
 * ------------------------------------------------------------------------ */

#define IQ_STATIC_MAX_TOKENS 2048

iq_status iq_prepare_q_static(const void* latent_bf16, int M,
                              const void* wq_e4m3, const uint8_t* wq_sf,
                              const int32_t* positions,
                              uint8_t* q_fp4, uint8_t* q_sf, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Indexer-Q preparation on host-resident tokens.  The pages have no
 * counterpart of this call; it serves a caller whose token rows and results
 * live in host memory (an offload or batch job), and overlaps their transfer
 * with the computation.  Same operation, arguments and results as
 * iq_prepare_q_ex, except where the buffers live:
 *
 *   latent_bf16 [M, 1536] BF16, positions [M] int32   -- read
 *   q_fp4 [M, 4096] uint8, q_sf [M, iq_fp4_scale_bytes(fp4_format)] uint8
 *                                                     -- written
 *     page-locked host memory (cudaHostAlloc / cudaMallocHost, or
 *     cudaHostRegister), or device memory of the current device; the same
 *     row-major layouts and alignments as iq_prepare_q.
 *   wq_e4m3, wq_sf: device memory, as in iq_prepare_q.
 *   workspace: iq_prepare_q_host_workspace(M, fp4_format) bytes of device
 *     memory, 256-byte aligned, used until the call's work completes.
 *
 * The rows are processed in chunks of iq_host_chunk_rows() rows (fewer
 * chunks when M needs more than 64).  On internal streams of the device the
 * quantizer of chunk c reads the chunk's latent rows and positions directly
 * from host memory, the GEMM of chunk c runs once that is done, and chunk c's
 * FP4 codes and scales are copied to q_fp4 / q_sf once its GEMM is done; so
 * reading chunk c + 1, computing chunk c and returning chunk c - 1 overlap.
 *
 * Ordering: the work starts after everything enqueued on `stream` before the
 * call, and everything enqueued on `stream` after the call starts after all
 * of it, the copies into q_fp4 / q_sf included.  Synchronize `stream` (or an
 * event recorded on it after the call) before reading the results on the
 * host, and leave the inputs unchanged until then.
 *
 * Errors: those of iq_prepare_q_ex, and IQ_ERR_ARG when latent_bf16,
 * positions, q_fp4 or q_sf is pageable host memory or another device's
 * memory, or the workspace is NULL; IQ_ERR_WORKSPACE when ws_bytes is smaller
 * than iq_prepare_q_host_workspace(M, fp4_format).  M == 0 returns IQ_OK.
 *
 * The first call on a device creates three streams and 132 events there
 * (kept until the process exits); make it outside stream capture.  Calls on
 * one device enqueue one at a time (a lock) because they share those streams.
 * ------------------------------------------------------------------------ */

size_t iq_prepare_q_host_workspace(int M, int fp4_format);

iq_status iq_prepare_q_host(const void* latent_bf16, int M,
                            const void* wq_e4m3, const uint8_t* wq_sf,
                            const int32_t* positions, int fp4_format,
                            uint8_t* q_fp4, uint8_t* q_sf,
                            void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Rows per chunk of iq_prepare_q_host, rounded up to a multiple of 256 and
 * clamped to [256, 2^20]; returns the previous value (default 1024). */
int iq_set_host_chunk_rows(int rows);
int iq_host_chunk_rows(void);

/* ------------------------------------------------------------------------
 * 3. The consumer of the prepared Q: the sparse-attention indexer's scores
 *    and top-k key selection (the TokenSpeed PR names the indexer top-k and
 *    writes it straight to its destination -- Summary; Prefill host-sync
 *    cleanup -- but gives neither formula nor layout; these are this
 *    library's readings).
 *
 *   score  I[t, s] = sum over heads h < 64 of w[t, h] * max(0, q(t, h) . k(s))
 *          q(t, h): head h of query token t, decoded from the MXFP4 Q that
 *            iq_prepare_q writes (q_fp4 [M, 4096], q_sf [M, 256]);
 *          k(s): the 128-dim key of cached token s, in the same MXFP4 format
 *            (k_fp4 [N, 64] bytes: element 2i in the low nibble of byte i;
 *            k_sf [N, 4] UE8M0 bytes, byte b for dims 32 b .. 32 b + 31);
 *          w: float32 [M, 64] per-head weights of each query token;
 *          keys s < L[t] are visible to query t (L: int32 [M], clamped to
 *            [0, N]; causal prefill passes position + 1).
 *   The head dot products are accumulated in float32 by the tensor cores;
 *   the ReLU and the weighted head sum are float32.
 * ------------------------------------------------------------------------ */

/* Writes logits[t * ld_logits + s] = I[t, s] for every visible pair (s <
 * L[t]); entries s >= L[t] are not written.  One kernel launch.
 * Requirements: M, N >= 0 (M == 0 or N == 0: IQ_OK, no launch); ld_logits >=
 * N; q_fp4, q_sf, k_fp4, k_sf and weights 16-byte aligned, lengths and
 * logits 4-byte aligned (else IQ_ERR_ALIGN); M * 64 < 2^31 (else IQ_ERR_ARG).
 * Launched as a programmatic dependent of the preceding kernel: nothing is
 * read before that kernel completes. */
iq_status iq_indexer_logits(const uint8_t* q_fp4, const uint8_t* q_sf, int M, const uint8_t* k_fp4,
                            const uint8_t* k_sf, int N, const float* weights, const int32_t* lengths,
                            float* logits, long long ld_logits, cudaStream_t stream);

/* For every query row t: the k visible keys (s < L[t]) with the largest
 * logits[t * ld_logits + s], ties to the smaller index (-0 and +0 tie), as
 * int32 indices in ascending order in indices[t * k .. t * k + k - 1], padded
 * with -1 when fewer than k keys are visible.  Scores must not be NaN.  One
 * kernel launch (one block per row), a programmatic dependent of the
 * preceding kernel (normally iq_indexer_logits).  Requirements: k >= 1,
 * ld_logits >= N, 4-byte aligned pointers. */
iq_status iq_indexer_topk(const float* logits, long long ld_logits, int M, int N, const int32_t* lengths, int k,
                          int32_t* indices, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* IQ_H_ */
