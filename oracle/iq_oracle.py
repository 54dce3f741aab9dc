"""CPU oracle for the DeepSeek-V4 indexer-Q preparation path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
this module: only the tests, the smoke check and the benchmark's CPU-baseline
leg use it.  It is plain numpy in float64, written to be read against the pages
it follows, with no blocking, fusion or reordering beyond what each definition
states.  It shares no code with the CUDA path.

Sources (cited by title and section):
  [TS]  TokenSpeed PR "perf(deepseek-v4): accelerate indexer Q and packed FP8
        quantization" -- Summary, Risk and fallback, Main-rebase compatibility fix.
  [TRT] TensorRT-LLM PR "Fuse DeepSeek-V4 Indexer Q projection with CuTe DSL"
        -- Walkthrough / sequence diagram, the review comment on
        dense_blockscaled_gemm_act_fusion.py (MXF8 sf_vec_size=32, 128-column
        tile), Description "Paths compared" (RoPE kernel, fusedCat FP4 kernel,
        output scale copies).
  [OCP] OCP Microscaling Formats (MX) v1.0 and OCP 8-bit Floating Point
        (E4M3 / E2M1 element formats, E8M0 scales) -- the element encodings the
        pages name (E4M3, E2M1, UE8M0) without restating them.

Readings where the pages are silent (named A1..A10 in the design notes):
  A1/A8  the "tiny-scale floor" is a floor of 1e-4 on the block amax, for the
         FP8 and the FP4 stage alike;
  A2     the sign of zero is kept (-0 encodes as the sign bit alone);
  A3     packed FP8 scales: int32 word [g][m] (g = block // 4, M-major, M padded
         to a multiple of 4), byte j of word g = scale of block 4g+j; pads 0;
  A4     W_q codes row-major [8192, 1536], UE8M0 scale bytes [64][12] per
         128x128 block;
  A5     the GEMM result is not rounded to BF16 before the epilogue;
  A6     NeoX RoPE on dims 0..63 of each head, pairs (i, i+32), theta = 10000;
  A7     Sylvester-ordered Hadamard-128 scaled by 1/sqrt(128), applied to the
         whole head after RoPE;
  A9     UE8M0 exponent = smallest e with qmax * 2^e >= floored amax (the same
         rule for FP8, qmax 448, and FP4, qmax 6);
  A10    FP4 packing: element 2i in the low nibble of byte i; FP4 scales
         [M][64 heads][4 blocks] bytes.
  The FP4 rounding decision is taken on the pre-quant value rounded to float32,
  the precision the CUDA path decides in.

FP4 output variants (the pages fix only MXFP4 with UE8M0 scales; these are the
alternatives the design notes list, each selectable on the CUDA path):
  "mx"      the rule above (A9: ceil, never saturates);
  "mx_ocp"  [OCP] MX v1.0 shared-scale rule: X = 2^(floor(log2 amax) - emax)
            with emax = 2 for E2M1, elements saturating at 6 (A13);
  "nv"      NVFP4-style: 1x16 blocks, the scale an E4M3 value (A14): per-tensor
            scale 1; s = E4M3 round-to-nearest of float32(amax / 6), raised
            to 2^-9 (the smallest positive E4M3) when it rounds to zero; codes
            E2M1(float32(z * float32(1 / s))); scales [M][64][8] E4M3 bytes.

Parity of A1, A8 and A9 (the absolute scale choices) is pinned only by these
readings: the pages do not state them.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E2M1_MAX = 6.0
AMAX_FLOOR = 1e-4          # A1 / A8
FP8_BLOCK = 128            # 1x128 activation blocks [TS] Summary; [TRT] Walkthrough
FP4_BLOCK = 32             # MXF8 sf_vec_size = 32 [TRT] review comment
NVFP4_BLOCK = 16           # A14
E4M3_MIN_POS = 2.0 ** -9   # smallest positive E4M3 value [OCP]
FP4_FORMATS = ("mx", "mx_ocp", "nv")
HEAD_DIM = 128
ROPE_DIM = 64
ROPE_THETA = 10000.0
UE8M0_BIAS = 127


# ---------------------------------------------------------------- formats [OCP]

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float64 (exact): BF16 is the top half of a float32."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):   # NaN patterns stay NaN
        return u.view(np.float32).astype(np.float64)


def e4m3_value_table() -> np.ndarray:
    """The 256 E4M3 (fn) code values: sign bit 7, exponent bits 6..3 with bias
    7, mantissa bits 2..0; exponent field 0 is subnormal (m/8 * 2^-6); codes
    0x7F and 0xFF are NaN and there is no infinity [OCP]."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        ef = (code >> 3) & 0xF
        m = code & 0x7
        if ef == 0xF and m == 0x7:
            vals[code] = np.nan
        elif ef == 0:
            vals[code] = s * (m / 8.0) * 2.0 ** -6
        else:
            vals[code] = s * (1.0 + m / 8.0) * 2.0 ** (ef - 7)
    return vals


def e2m1_value_table() -> np.ndarray:
    """The 16 E2M1 code values: sign bit 3, exponent bits 2..1 with bias 1,
    mantissa bit 0; exponent field 0 is subnormal (m/2) [OCP]."""
    vals = np.empty(16, dtype=np.float64)
    for code in range(16):
        s = -1.0 if code & 0x8 else 1.0
        ef = (code >> 1) & 0x3
        m = code & 0x1
        vals[code] = s * (m / 2.0 if ef == 0 else (1.0 + m / 2.0) * 2.0 ** (ef - 1))
    return vals


_E4M3 = e4m3_value_table()
_E2M1 = e2m1_value_table()
_E4M3_POS = _E4M3[:0x7F]   # codes 0x00..0x7E, strictly increasing
_E2M1_POS = _E2M1[:8]      # codes 0..7, strictly increasing


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    return _E4M3[np.asarray(codes, dtype=np.uint8)]


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    return _E2M1[np.asarray(codes, dtype=np.uint8) & 0xF]


def decode_ue8m0(b: np.ndarray) -> np.ndarray:
    """UE8M0 byte b encodes 2^(b - 127) [OCP]."""
    return np.ldexp(1.0, np.asarray(b, dtype=np.int64) - UE8M0_BIAS)


def _round_to_grid(v: np.ndarray, min_normal_exp: int, mant_bits: int, vmax: float) -> np.ndarray:
    """Round |v| to nearest, ties to even, on a binary grid with ``mant_bits``
    stored mantissa bits and subnormals below 2^min_normal_exp; saturate to vmax.
    The step in binade 2^E is 2^(E - mant_bits); a / step is exact."""
    a = np.abs(v)
    _, ex = np.frexp(a)                        # a = f * 2^ex, f in [0.5, 1)
    E = np.maximum(ex.astype(np.int64) - 1, min_normal_exp)
    step = np.ldexp(1.0, E - mant_bits)
    q = np.rint(a / step) * step               # np.rint rounds half to even
    return np.minimum(q, vmax)


def round_to_e4m3_codes(v: np.ndarray) -> np.ndarray:
    """E4M3 code of round-to-nearest-even(v), saturating at 448, sign kept (A2)."""
    v = np.asarray(v, dtype=np.float64)
    q = _round_to_grid(v, -6, 3, E4M3_MAX)
    idx = np.searchsorted(_E4M3_POS, q)
    assert np.array_equal(_E4M3_POS[idx], q)
    return (idx | (np.signbit(v).astype(np.int64) << 7)).astype(np.uint8)


def round_to_e2m1_codes(v: np.ndarray) -> np.ndarray:
    """E2M1 code of round-to-nearest-even(v), saturating at 6, sign kept (A2)."""
    v = np.asarray(v, dtype=np.float64)
    q = _round_to_grid(v, 0, 1, E2M1_MAX)
    idx = np.searchsorted(_E2M1_POS, q)
    assert np.array_equal(_E2M1_POS[idx], q)
    return (idx | (np.signbit(v).astype(np.int64) << 3)).astype(np.uint8)


def ue8m0_exponent(amax: np.ndarray, qmax: float, floor: float = AMAX_FLOOR) -> np.ndarray:
    """Power-of-two scale exponent of a block (A1, A8, A9): the smallest integer
    e with qmax * 2^e >= max(amax, floor).  [TS] Risk and fallback names the
    floor; the ceil rule makes the block's largest magnitude land in
    (qmax/2, qmax] after division by 2^e."""
    a = np.maximum(np.asarray(amax, dtype=np.float64), floor)
    e = np.ceil(np.log2(a / qmax)).astype(np.int64)
    # log2 may be one ulp off next to a power of two: settle e exactly.
    e = np.where(np.ldexp(qmax, e - 1) >= a, e - 1, e)
    e = np.where(np.ldexp(qmax, e) < a, e + 1, e)
    return e


# -------------------------------------------------- stage 1: FP8 1x128 quantizer

def quantize_fp8_1x128(x: np.ndarray):
    """Per row and per 1x128 block: amax, floor, UE8M0 exponent, E4M3 codes of
    x * 2^-e ([TS] Summary "packed-UE8M0 FP8 online quantizer" and Risk and
    fallback; [TRT] Walkthrough "create FP8 input and UE8M0 scales").

    x: float64 [M, K], K % 128 == 0.  Returns (codes uint8 [M, K], scale bytes
    uint8 [M, K/128])."""
    M, K = x.shape
    assert K % FP8_BLOCK == 0
    blocks = x.reshape(M, K // FP8_BLOCK, FP8_BLOCK)
    amax = np.abs(blocks).max(axis=2) if M else np.zeros((0, K // FP8_BLOCK))
    e = ue8m0_exponent(amax, E4M3_MAX)
    scaled = blocks * np.ldexp(1.0, -e)[..., None]        # exact power-of-two scaling
    codes = round_to_e4m3_codes(scaled).reshape(M, K)
    return codes, (e + UE8M0_BIAS).astype(np.uint8)


def pack_scales_m_major(scale_bytes: np.ndarray) -> np.ndarray:
    """Packed UE8M0 scale contract (A3): int32 words [ceil(nb/4)][align4(M)],
    byte j (little-endian) of word [g][m] is the scale of block 4g+j of row m;
    rows m >= M and bytes past the last block are zero."""
    M, nb = scale_bytes.shape
    G = -(-nb // 4)
    m_al = (M + 3) // 4 * 4
    words = np.zeros((G, m_al), dtype=np.uint32)
    for kb in range(nb):
        words[kb // 4, :M] |= scale_bytes[:, kb].astype(np.uint32) << np.uint32(8 * (kb % 4))
    return words.view(np.int32)


def fp8_quant_1x128_ue8m0(x_bits: np.ndarray):
    """The first call of the library: BF16 bits [M, K] -> (E4M3 codes [M, K],
    packed scale words [ceil(K/512)][align4(M)] int32)."""
    codes, sb = quantize_fp8_1x128(bf16_bits_to_f64(x_bits))
    return codes, pack_scales_m_major(sb)


# -------------------------------------------- stage 2: block-scaled FP8 GEMM

def block_scaled_gemm(xq: np.ndarray, x_sb: np.ndarray, wq: np.ndarray, w_sb: np.ndarray) -> np.ndarray:
    """Y[m, n] = sum over 128-blocks kb of 2^(eX[m,kb] + eW[n/128,kb]) *
    sum_{k in kb} x[m,k] * w[n,k], on decoded E4M3 values ([TRT] Walkthrough:
    FP8 GEMM on the FP8 input and UE8M0 scales; A4, A5).

    Each per-block partial sum of E4M3 products is exact in float64, so the
    result is exact up to the float64 rounding of the 12-term outer sum."""
    M, K = xq.shape
    N = wq.shape[0]
    X = decode_e4m3(xq)
    W = decode_e4m3(wq)
    sx = decode_ue8m0(x_sb)                                  # [M, K/128]
    sw = np.repeat(decode_ue8m0(w_sb), FP8_BLOCK, axis=0)    # [N, K/128]
    Y = np.zeros((M, N), dtype=np.float64)
    for kb in range(K // FP8_BLOCK):
        sl = slice(kb * FP8_BLOCK, (kb + 1) * FP8_BLOCK)
        Y += (X[:, sl] @ W[:, sl].T) * sx[:, kb:kb + 1] * sw[:, kb][None, :]
    return Y


# ------------------------------------------------------------------ RoPE (A6)

def rope_inv_freq() -> np.ndarray:
    """theta^(-2i/64) for i = 0..31."""
    i = np.arange(ROPE_DIM // 2, dtype=np.float64)
    return ROPE_THETA ** (-2.0 * i / ROPE_DIM)


def rope_neox(Y: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """NeoX rotation of dims 0..63 of every 128-dim head by pos * theta^(-2i/64)
    ([TS] Summary and [TRT] Paths compared: the MLA RoPE kernel on the rope
    slice of the indexer Q).  Pairs (i, i+32):
        r_i      = q_i c - q_{i+32} s
        r_{i+32} = q_{i+32} c + q_i s
    dims 64..127 pass through."""
    M = Y.shape[0]
    Yh = Y.reshape(M, -1, HEAD_DIM).copy()
    ang = np.asarray(pos, dtype=np.float64)[:, None] * rope_inv_freq()[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    half = ROPE_DIM // 2
    x1 = Yh[:, :, :half].copy()
    x2 = Yh[:, :, half:ROPE_DIM].copy()
    Yh[:, :, :half] = x1 * c - x2 * s
    Yh[:, :, half:ROPE_DIM] = x2 * c + x1 * s
    return Yh.reshape(M, -1)


# -------------------------------------------------------------- Hadamard (A7)

def hadamard_matrix(n: int = HEAD_DIM) -> np.ndarray:
    """Sylvester Hadamard matrix H[i][j] = (-1)^popcount(i & j)."""
    i = np.arange(n)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1.0, -1.0)


def hadamard_heads(R: np.ndarray) -> np.ndarray:
    """z = H_128 r / sqrt(128) for every head ([TS] Summary and Main-rebase
    compatibility fix: the Hadamard transform of the indexer Q)."""
    M = R.shape[0]
    H = hadamard_matrix(HEAD_DIM)
    Z = R.reshape(M, -1, HEAD_DIM) @ H.T / np.sqrt(HEAD_DIM)
    return Z.reshape(M, -1)


# ------------------------------------------------------- FP4 (A8, A9, A10)

def quantize_fp4_1x32(z: np.ndarray):
    """Per 1x32 block: amax, floor, UE8M0 exponent (qmax 6), E2M1 codes of
    z * 2^-e ([TS] Summary "fusedCat FP4"; [TRT] review comment: MXF8
    sf_vec_size = 32).  Returns (codes uint8 [M, D] one code per element,
    scale bytes uint8 [M, D/32])."""
    M, D = z.shape
    b = z.reshape(M, D // FP4_BLOCK, FP4_BLOCK)
    amax = np.abs(b).max(axis=2) if M else np.zeros((0, D // FP4_BLOCK))
    e = ue8m0_exponent(amax, E2M1_MAX)
    codes = round_to_e2m1_codes(b * np.ldexp(1.0, -e)[..., None])
    return codes.reshape(M, D), (e + UE8M0_BIAS).astype(np.uint8)


def ue8m0_exponent_ocp(amax: np.ndarray, floor: float = AMAX_FLOOR) -> np.ndarray:
    """[OCP] MX v1.0 shared scale of an E2M1 block (A13): X = 2^e with
    e = floor(log2(max(amax, floor))) - 2, emax(E2M1) = 2, so the block's
    largest magnitude lands in [4, 8) before the elements saturate at 6."""
    a = np.maximum(np.asarray(amax, dtype=np.float64), floor)
    _, ex = np.frexp(a)                          # a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
    return ex.astype(np.int64) - 1 - 2


def quantize_fp4_1x32_ocp(z: np.ndarray):
    """quantize_fp4_1x32 with the [OCP] floor rule (A13).  Returns (codes
    uint8 [M, D], scale bytes uint8 [M, D/32])."""
    M, D = z.shape
    b = z.reshape(M, D // FP4_BLOCK, FP4_BLOCK)
    amax = np.abs(b).max(axis=2) if M else np.zeros((0, D // FP4_BLOCK))
    e = ue8m0_exponent_ocp(amax)
    codes = round_to_e2m1_codes(b * np.ldexp(1.0, -e)[..., None])
    return codes.reshape(M, D), (e + UE8M0_BIAS).astype(np.uint8)


def nvfp4_block_scale(amax_f32: np.ndarray) -> np.ndarray:
    """E4M3 scale code of an NVFP4 block (A14): round-to-nearest-even of
    float32(max(amax, floor) / 6) onto E4M3, or 2^-9 when that is zero."""
    a = np.maximum(np.asarray(amax_f32, dtype=np.float32), np.float32(AMAX_FLOOR))
    s = (a / np.float32(E2M1_MAX)).astype(np.float64)          # float32 division, then exact in float64
    code = round_to_e4m3_codes(s)
    return np.where(code == 0, np.uint8(1), code).astype(np.uint8)   # code 1 = 2^-9


def quantize_nvfp4_1x16(z_f32: np.ndarray):
    """NVFP4-style 1x16 blocks with E4M3 scales (A14) on float32 values.
    Returns (codes uint8 [M, D], scale codes uint8 [M, D/16])."""
    M, D = z_f32.shape
    b = np.asarray(z_f32, dtype=np.float32).reshape(M, D // NVFP4_BLOCK, NVFP4_BLOCK)
    amax = np.abs(b).max(axis=2) if M else np.zeros((0, D // NVFP4_BLOCK), np.float32)
    sc = nvfp4_block_scale(amax)
    r = (1.0 / decode_e4m3(sc)).astype(np.float32)           # float32(1 / s), correctly rounded
    u = (b * r[..., None]).astype(np.float32)                 # float32 product
    codes = round_to_e2m1_codes(u.astype(np.float64))
    return codes.reshape(M, D), sc


def pack_fp4(codes: np.ndarray) -> np.ndarray:
    """Two E2M1 codes per byte, element 2i in the low nibble (A10)."""
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


# ----------------------------------------------------------------- the chain

def prepare_q(latent_bits: np.ndarray, wq: np.ndarray, w_sb: np.ndarray, pos: np.ndarray, fmt: str = "mx"):
    """The second call of the library, end to end ([TRT] sequence diagram:
    quantize the latent to FP8 with UE8M0 scales, block-scaled GEMM with the
    RoPE and FP4 epilogue, return packed FP4 Q and scales).  fmt picks the FP4
    output variant (module docstring).

    Returns (q_fp4 uint8 [M, 4096], q_sf uint8 [M, 256] ([M, 512] for "nv"),
    z float64 [M, 8192]) where z is the pre-quant Q (after RoPE and
    Hadamard)."""
    x = bf16_bits_to_f64(latent_bits)
    xq, x_sb = quantize_fp8_1x128(x)
    y = block_scaled_gemm(xq, x_sb, wq, w_sb)
    z = hadamard_heads(rope_neox(y, pos))
    z_decide = z.astype(np.float32).astype(np.float64)   # decision precision: float32
    if fmt == "mx":
        codes, q_sf = quantize_fp4_1x32(z_decide)
    elif fmt == "mx_ocp":
        codes, q_sf = quantize_fp4_1x32_ocp(z_decide)
    elif fmt == "nv":
        codes, q_sf = quantize_nvfp4_1x16(z_decide.astype(np.float32))
    else:
        raise ValueError(f"unknown FP4 format {fmt!r}")
    return pack_fp4(codes), q_sf, z


def prequant_q_rows(latent_bits: np.ndarray, wq: np.ndarray, w_sb: np.ndarray,
                    pos: np.ndarray, rows: np.ndarray, fmt: str = "mx"):
    """prepare_q on a subset of rows (rows are independent), for sampled checks
    of large problems."""
    rows = np.asarray(rows)
    return prepare_q(latent_bits[rows], wq, w_sb, pos[rows], fmt)


# ------------------------------------------- downstream: indexer logits, top-k
# The consumer of the prepared Q: the sparse-attention indexer's score of
# every (query token, cached key) pair and the selection of the top-k keys per
# query ([TS] Summary and Prefill host-sync cleanup: the indexer top-k written
# straight to its destination).  The pages name this consumer but not its
# formulas or layouts; the readings (A17-A22 in the design notes):
#   A17  score I[t, s] = sum_h w[t, h] * max(0, q(t, h) . k(s)) over the 64
#        heads, q(t, h) the decoded head h of token t's FP4 Q, k(s) the decoded
#        128-dim key of token s (one key per token, shared by all heads);
#   A18  the key cache is MXFP4 like Q: codes [N, 64] bytes (element 2i in the
#        low nibble of byte i), UE8M0 scale bytes [N, 4] (one per 32 dims);
#   A19  w: float32 [M, 64], given;
#   A20  query t sees keys s < L[t] (L: int32 [M]); the others score -inf;
#   A21  top-k: the k visible keys with the largest scores, ties to the
#        smaller key index, written as int32 indices in ascending order and
#        padded with -1 when fewer than k keys are visible;
#   A22  the decision precision: the oracle scores in float64 from the decoded
#        values (each head's dot product is exact there).

INDEXER_HEADS = 64


def decode_mxfp4(codes_packed: np.ndarray, scale_bytes: np.ndarray, block: int = FP4_BLOCK) -> np.ndarray:
    """Packed E2M1 codes [R, D/2] (element 2i in the low nibble of byte i,
    A10/A18) and UE8M0 scale bytes [R, D/block] -> float64 [R, D]."""
    c = np.asarray(codes_packed, dtype=np.uint8)
    R = c.shape[0]
    codes = np.empty((R, c.shape[1] * 2), dtype=np.uint8)
    codes[:, 0::2] = c & 0xF
    codes[:, 1::2] = c >> 4
    v = decode_e2m1(codes).reshape(R, -1, block)
    return (v * decode_ue8m0(scale_bytes)[..., None]).reshape(R, -1)


def indexer_logits(q_fp4: np.ndarray, q_sf: np.ndarray, k_fp4: np.ndarray, k_sf: np.ndarray,
                   weights: np.ndarray, lengths: np.ndarray) -> np.ndarray:
    """I[t, s] = sum_h w[t, h] max(0, q(t, h) . k(s)) for s < L[t], -inf
    otherwise (A17-A20).  q_fp4 [M, 4096] / q_sf [M, 256] as iq_prepare_q
    writes them, k_fp4 [N, 64] / k_sf [N, 4], weights [M, 64], lengths [M].
    Returns float64 [M, N]."""
    M = q_fp4.shape[0]
    N = k_fp4.shape[0]
    Q = decode_mxfp4(q_fp4.reshape(M * INDEXER_HEADS, HEAD_DIM // 2),
                     q_sf.reshape(M * INDEXER_HEADS, HEAD_DIM // FP4_BLOCK)).reshape(M, INDEXER_HEADS, HEAD_DIM)
    K = decode_mxfp4(k_fp4, k_sf)                                   # [N, 128]
    dots = np.einsum("mhd,nd->mhn", Q, K)                           # exact per head (dyadic values)
    scores = np.einsum("mh,mhn->mn", np.asarray(weights, np.float64), np.maximum(dots, 0.0))
    visible = np.arange(N)[None, :] < np.asarray(lengths, np.int64)[:, None]
    return np.where(visible, scores, -np.inf)


def indexer_logit_magnitude(q_fp4, q_sf, k_fp4, k_sf, weights) -> np.ndarray:
    """S[t, s] = sum_h |w[t, h]| sum_d |q(t, h, d) k(s, d)|: the sum of the
    magnitudes of every term of I[t, s], which bounds the rounding error of
    forming I in float32 (A22)."""
    M = q_fp4.shape[0]
    Q = np.abs(decode_mxfp4(q_fp4.reshape(M * INDEXER_HEADS, HEAD_DIM // 2),
                            q_sf.reshape(M * INDEXER_HEADS, HEAD_DIM // FP4_BLOCK))).reshape(M, INDEXER_HEADS, HEAD_DIM)
    K = np.abs(decode_mxfp4(k_fp4, k_sf))
    return np.einsum("mh,mhn->mn", np.abs(np.asarray(weights, np.float64)), np.einsum("mhd,nd->mhn", Q, K))


def indexer_topk(scores: np.ndarray, lengths: np.ndarray, k: int) -> np.ndarray:
    """A21: per row t, the k keys s < L[t] with the largest scores (ties to
    the smaller index), as int32 indices in ascending order, -1 padded."""
    M = scores.shape[0]
    out = np.full((M, k), -1, dtype=np.int32)
    for t in range(M):
        L = int(min(max(lengths[t], 0), scores.shape[1]))
        idx = np.arange(L)
        order = np.lexsort((idx, -np.asarray(scores[t, :L], np.float64)))   # score descending, then index
        chosen = np.sort(order[:k])
        out[t, :len(chosen)] = chosen
    return out
