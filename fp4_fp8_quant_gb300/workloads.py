"""Seeded synthetic inputs for the indexer-Q preparation path.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It holds input recipes only: random draws, the BF16 storage
format of the activations, and a library cast (torch's float8_e4m3fn) that
turns Gaussian draws into weight codes.  None of the quantizer, GEMM, RoPE,
Hadamard or FP4 arithmetic lives here.

Shapes follow the DeepSeek-V4 indexer as the TensorRT-LLM PR "Fuse DeepSeek-V4
Indexer Q projection with CuTe DSL" wires it (Walkthrough: the indexer-Q
projection from the latent into 64 heads of 128 dims) and the TokenSpeed PR
"perf(deepseek-v4): accelerate indexer Q and packed FP8 quantization"
(Performance: 128 and 4,632 token microbenchmarks).  Every generator uses
numpy's PCG64 so that the same seed gives the same bytes on every host.
"""

from __future__ import annotations

import numpy as np

LATENT_DIM = 1536          # K of the indexer-Q projection
N_HEADS = 64
HEAD_DIM = 128
Q_DIM = N_HEADS * HEAD_DIM  # 8192
MAX_POSITION = 163840       # positions are drawn from [0, MAX_POSITION)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Store float32 values as BF16 bit patterns (round to nearest even).

    This is the storage format of the synthetic activations, not a step of the
    method: the method starts from BF16 inputs.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def latent(M: int, K: int = LATENT_DIM, seed: int = 0,
           outlier_p: float = 0.001, outlier_scale: float = 50.0) -> np.ndarray:
    """BF16 bits [M, K]: N(0,1) with each element independently scaled by
    ``outlier_scale`` with probability ``outlier_p``."""
    rng = _rng(seed)
    x = rng.standard_normal((M, K), dtype=np.float32)
    if outlier_p > 0:
        hit = rng.random((M, K)) < outlier_p
        x = np.where(hit, x * np.float32(outlier_scale), x)
    return f32_to_bf16_bits(x)


def quant_blocks_input(M: int, K: int = 7168, seed: int = 1,
                       p_large: float = 0.01, large_scale: float = 1e3,
                       p_zero: float = 0.01, p_tiny: float = 0.01) -> np.ndarray:
    """BF16 bits [M, K] for the stand-alone quantizer workload.

    N(0,1) data; one uniform draw per 1x128 block picks its class:
    ``p_large`` of blocks are scaled by ``large_scale``, ``p_zero`` are all
    zero and ``p_tiny`` hold N(0,1)*1e-7 clipped to |x| < 9e-7, so that their
    amax sits below 1e-6 and the tiny-scale floor decides their scale.
    """
    assert K % 128 == 0
    rng = _rng(seed)
    x = rng.standard_normal((M, K), dtype=np.float32)
    u = rng.random((M, K // 128))
    xb = x.reshape(M, K // 128, 128)
    large = u < p_large
    zero = (u >= p_large) & (u < p_large + p_zero)
    tiny = (u >= p_large + p_zero) & (u < p_large + p_zero + p_tiny)
    xb[large] *= np.float32(large_scale)
    xb[zero] = 0.0
    xb[tiny] = np.clip(xb[tiny] * np.float32(1e-7), np.float32(-8.9e-7), np.float32(8.9e-7))
    return f32_to_bf16_bits(xb.reshape(M, K))


def weights(seed: int = 0, N: int = Q_DIM, K: int = LATENT_DIM):
    """Indexer-Q weight as E4M3 codes [N, K] (row-major, one row per output
    feature) and UE8M0 block-scale bytes [N/128, K/128].

    The codes are torch's float8_e4m3fn cast of N(0,1)*100 draws clipped to the
    E4M3 range; each 128x128 block takes exponent -12 + U{-1,0,1}, so W is close
    to N(0, 0.02) with power-of-two block scales.
    """
    import torch
    rng = _rng(1000 + seed)
    v = np.clip(rng.standard_normal((N, K), dtype=np.float32) * np.float32(100.0), -448.0, 448.0)
    codes = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    exps = -12 + rng.integers(-1, 2, size=(N // 128, K // 128))
    sf = (exps + 127).astype(np.uint8)
    return codes, sf


SWEEP_ROW_BLOCK = 256        # rows per independently seeded block of the large inputs


def sweep_quant_block(M: int, K: int, block: int, seed: int = 4,
                      outlier_p: float = 0.005, outlier_scale: float = 100.0) -> np.ndarray:
    """BF16 bits of rows [256 * block, min(M, 256 * (block + 1))) of the
    stand-alone quantizer input of the long-prefill sweep ([M, K], N(0,1) with
    0.5% of elements x100).  Each 256-row block has its own seeded stream, so a
    sample of rows can be regenerated without the whole matrix (which reaches
    65536 x 7168 elements)."""
    r0 = block * SWEEP_ROW_BLOCK
    rows = min(M, r0 + SWEEP_ROW_BLOCK) - r0
    rng = np.random.Generator(np.random.PCG64([seed, block, K]))
    x = rng.standard_normal((rows, K), dtype=np.float32)
    hit = rng.random((rows, K), dtype=np.float32) < np.float32(outlier_p)
    x = np.where(hit, x * np.float32(outlier_scale), x)
    return f32_to_bf16_bits(x)


def sweep_quant_rows(M: int, K: int, rows, seed: int = 4) -> np.ndarray:
    """The given rows of the same input (BF16 bits [len(rows), K])."""
    rows = np.asarray(rows)
    out = np.empty((len(rows), K), np.uint16)
    for b in np.unique(rows // SWEEP_ROW_BLOCK):
        blk = sweep_quant_block(M, K, int(b), seed)
        sel = rows // SWEEP_ROW_BLOCK == b
        out[sel] = blk[rows[sel] - int(b) * SWEEP_ROW_BLOCK]
    return out


def positions(M: int, seed: int = 0, contiguous: bool = False) -> np.ndarray:
    """int32 [M] token positions: 0..M-1, or uniform in [0, MAX_POSITION)."""
    if contiguous:
        return np.arange(M, dtype=np.int32)
    return _rng(2000 + seed).integers(0, MAX_POSITION, size=M, dtype=np.int64).astype(np.int32)


# Named workloads (sizes and distributions of the indexer-Q path).
def chain_workload(M: int, seed: int, outlier_p: float, outlier_scale: float,
                   contiguous_positions: bool = False):
    """Latent bits, weight codes, weight scale bytes and positions for one
    indexer-Q chain problem."""
    x = latent(M, LATENT_DIM, seed=seed, outlier_p=outlier_p, outlier_scale=outlier_scale)
    wq, wsf = weights(seed=0)
    pos = positions(M, seed=seed, contiguous=contiguous_positions)
    return x, wq, wsf, pos


def tiny_chain(M: int = 16, seed: int = 0):
    """16-token chain: N(0,1) latent with 0.1% outliers x50, random positions."""
    return chain_workload(M, seed, 0.001, 50.0)


def prefill_chain(M: int = 4632, seed: int = 3):
    """4,632-token prefill chain: 0.1% outliers x50, positions 0..M-1."""
    return chain_workload(M, seed, 0.001, 50.0, contiguous_positions=True)


def sweep_chain(M: int, seed: int = 4):
    """Long-prefill sweep point: 0.5% outliers x100, random positions."""
    return chain_workload(M, seed, 0.005, 100.0)


def decode_chain(M: int, seed: int = 2):
    """Decode batch of M tokens: plain N(0,1) latent, random positions."""
    return chain_workload(M, seed, 0.0, 1.0)


# Inputs of the downstream indexer consumer (logits and top-k).
_FP4_MAGNITUDE_P = np.array([0.22, 0.2, 0.16, 0.14, 0.1, 0.08, 0.06, 0.04])   # codes 0..7


def mxfp4_codes(rows: int, dims: int, rng: np.random.Generator) -> np.ndarray:
    """Packed E2M1 codes [rows, dims / 2] (element 2i in the low nibble):
    magnitude codes drawn from a fixed distribution favouring small values,
    random signs.  A draw of codes, not a quantization of anything."""
    mag = rng.choice(8, size=(rows, dims), p=_FP4_MAGNITUDE_P).astype(np.uint8)
    sign = (rng.random((rows, dims)) < 0.5).astype(np.uint8) << 3
    c = mag | sign
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def indexer_inputs(M: int, N: int, seed: int = 0, causal: bool = True):
    """Query side [M, 4096] codes + [M, 256] UE8M0 scale bytes (the layout
    iq_prepare_q writes), key cache [N, 64] codes + [N, 4] scale bytes, per-head
    weights float32 [M, 64] N(0, 1/64), and visible lengths int32 [M]: the M
    queries are the last M positions of an N-token sequence (L = position + 1)
    when causal, else every key is visible."""
    rng = _rng(3000 + seed)
    q = mxfp4_codes(M * N_HEADS, HEAD_DIM, rng).reshape(M, Q_DIM // 2)
    q_sf = rng.integers(122, 127, size=(M, Q_DIM // 32)).astype(np.uint8)
    k = mxfp4_codes(N, HEAD_DIM, rng)
    k_sf = rng.integers(122, 127, size=(N, HEAD_DIM // 32)).astype(np.uint8)
    w = (rng.standard_normal((M, N_HEADS)) / 8).astype(np.float32)
    if causal:
        lengths = np.clip(np.arange(N - M, N) + 1, 0, N).astype(np.int32)
    else:
        lengths = np.full(M, N, np.int32)
    return q, q_sf, k, k_sf, w, lengths


def indexer_keys(N: int, seed: int = 0):
    """A key cache alone: codes [N, 64] and UE8M0 scale bytes [N, 4], drawn as
    in indexer_inputs."""
    rng = _rng(4000 + seed)
    return mxfp4_codes(N, HEAD_DIM, rng), rng.integers(122, 127, size=(N, HEAD_DIM // 32)).astype(np.uint8)


def indexer_weights(M: int, seed: int = 0) -> np.ndarray:
    """Per-head weights alone: float32 [M, 64], N(0, 1/64)."""
    return (_rng(5000 + seed).standard_normal((M, N_HEADS)) / 8).astype(np.float32)
