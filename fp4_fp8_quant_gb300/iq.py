"""Python binding of libiq (include/iq.h): ctypes argument marshalling only.

Every step of the path runs in the library's CUDA kernels.  PyTorch supplies
device memory and the current stream.  There is no fallback: if the library
has not been built, or the device is not sm_103, the calls raise.
"""

from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

LATENT_DIM = 1536
N_HEADS = 64
HEAD_DIM = 128
Q_DIM = 8192
SMALL_M_MAX = 128

_STATUS = {0: "IQ_OK", -1: "IQ_ERR_ARG", -2: "IQ_ERR_ALIGN", -3: "IQ_ERR_SHAPE", -4: "IQ_ERR_ARCH",
           -5: "IQ_ERR_CUDA", -6: "IQ_ERR_WORKSPACE", -7: "IQ_ERR_TIMEOUT"}

# Every symbol include/iq.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
SIGNATURES = {
    "iq_status_str": (ctypes.c_char_p, [_I]),
    "iq_device_status": (_I, [ctypes.POINTER(ctypes.c_uint32), _I]),
    "iq_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
    "iq_selftest_workspace": (_SZ, []),
    "iq_selftest_wait_timeout": (_I, [_P, _SZ, ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint32), _P]),
    "iq_debug_fail_next_setups": (None, [_I]),
    "iq_debug_e2m1_codes": (_I, [_P, ctypes.c_longlong, _P, _P]),
    "iq_fp8_scale_words": (_SZ, [_I, _I]),
    "iq_fp8_quant_1x128_ue8m0": (_I, [_P, _I, _I, _I, _P, _I, _P, _P]),
    "iq_prepare_q_workspace": (_SZ, [_I]),
    "iq_prepare_q": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "iq_prepare_q_debug": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "iq_gemm_rope_hadamard_fp4": (_I, [_P, _P, _I, _P, _P, _P, _P, _P, _P, _P]),
    "iq_prepare_q_static": (_I, [_P, _I, _P, _P, _P, _P, _P, _P]),
    "iq_set_small_m_threshold": (_I, [_I]),
    "iq_small_m_threshold": (_I, []),
    "iq_set_gemm_tiling": (None, [_I, _I]),
    "iq_set_quant_fusion": (_I, [_I]),
    "iq_debug_delay_quant_ns": (None, [ctypes.c_uint64]),
    "iq_fp4_scale_bytes": (_SZ, [_I]),
    "iq_prepare_q_ex": (_I, [_P, _I, _P, _P, _P, _I, _P, _P, _P, _P, _SZ, _P]),
    "iq_prepare_q_host_workspace": (_SZ, [_I, _I]),
    "iq_prepare_q_host": (_I, [_P, _I, _P, _P, _P, _I, _P, _P, _P, _SZ, _P]),
    "iq_set_host_chunk_rows": (_I, [_I]),
    "iq_host_chunk_rows": (_I, []),
    "iq_indexer_logits": (_I, [_P, _P, _I, _P, _P, _I, _P, _P, _P, ctypes.c_longlong, _P]),
    "iq_indexer_topk": (_I, [_P, ctypes.c_longlong, _I, _I, _P, _I, _P, _P]),
}

# FP4 output variants (include/iq.h, iq_fp4_format).
FP4_FORMATS = {"mx": 0, "mx_ocp": 1, "nv": 2}

_lib = None


class IQError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {_STATUS.get(code, code)} ({status_str(code)})")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded libiq.so.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libiq.so is not built ({LIB_PATH}); run python -m fp4_fp8_quant_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_str(code: int) -> str:
    try:
        return lib().iq_status_str(code).decode()
    except ImportError:
        return _STATUS.get(code, str(code))


def _check(code: int, what: str):
    if code != 0:
        raise IQError(code, what)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _require(t: torch.Tensor, name: str, dtypes, shape=None, contiguous=True):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_U8 = (torch.uint8, torch.float8_e4m3fn)


def scale_words(M: int, K: int) -> int:
    return int(lib().iq_fp8_scale_words(M, K))


def fp8_quant_1x128_ue8m0(x: torch.Tensor, y: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                          stream=None):
    """BF16 [M, K] (row stride may exceed K) -> (E4M3 codes uint8 [M, K],
    packed UE8M0 scales int32 [ceil(K/512), align4(M)])."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D tensor with unit column stride")
    _require(x, "x", (torch.bfloat16,), contiguous=False)
    M, K = x.shape
    if y is None:
        y = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((max(1, -(-K // 512)), (M + 3) // 4 * 4), dtype=torch.int32, device=x.device)
    if y.dim() != 2 or y.stride(1) != 1:
        raise ValueError("y must be a 2-D tensor with unit column stride")
    _require(y, "y", _U8, contiguous=False)
    _require(scales, "scales", (torch.int32,))
    _check(lib().iq_fp8_quant_1x128_ue8m0(_ptr(x), M, K, x.stride(0), _ptr(y), y.stride(0), _ptr(scales),
                                          _stream(stream)), "iq_fp8_quant_1x128_ue8m0")
    return y, scales


def prepare_q_workspace_bytes(M: int) -> int:
    return int(lib().iq_prepare_q_workspace(M))


def fp4_scale_bytes(fp4_format: str = "mx") -> int:
    """Scale bytes per token of an FP4 output variant (256 or 512)."""
    return int(lib().iq_fp4_scale_bytes(FP4_FORMATS[fp4_format]))


def _prepare_out(M, device, q_fp4, q_sf, fp4_format="mx"):
    sf_cols = Q_DIM // 16 if fp4_format == "nv" else Q_DIM // 32
    if q_fp4 is None:
        q_fp4 = torch.empty((M, Q_DIM // 2), dtype=torch.uint8, device=device)
    if q_sf is None:
        q_sf = torch.empty((M, sf_cols), dtype=torch.uint8, device=device)
    _require(q_fp4, "q_fp4", (torch.uint8,), (M, Q_DIM // 2))
    _require(q_sf, "q_sf", (torch.uint8,), (M, sf_cols))
    return q_fp4, q_sf


def prepare_q(latent: torch.Tensor, wq: torch.Tensor, wq_sf: torch.Tensor, positions: torch.Tensor, *,
              q_fp4: torch.Tensor | None = None, q_sf: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, q_prequant: torch.Tensor | None = None,
              debug: bool = False, fp4_format: str = "mx", stream=None):
    """Indexer-Q preparation: returns (q_fp4 uint8 [M, 4096], q_sf uint8
    [M, 256] ([M, 512] for fp4_format="nv")) and, with debug=True, also the
    float32 pre-quant Q [M, 8192].  fp4_format: "mx" (default), "mx_ocp" or
    "nv" (include/iq.h, FP4 output variants)."""
    M = latent.shape[0]
    if fp4_format not in FP4_FORMATS:
        raise ValueError(f"fp4_format must be one of {sorted(FP4_FORMATS)}")
    _require(latent, "latent", (torch.bfloat16,), (M, LATENT_DIM))
    _require(wq, "wq", _U8, (Q_DIM, LATENT_DIM))
    _require(wq_sf, "wq_sf", (torch.uint8,), (N_HEADS, LATENT_DIM // 128))
    _require(positions, "positions", (torch.int32,), (M,))
    q_fp4, q_sf = _prepare_out(M, latent.device, q_fp4, q_sf, fp4_format)
    ws_bytes = prepare_q_workspace_bytes(M)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=latent.device)
    _require(workspace, "workspace", (torch.uint8,))
    if debug and q_prequant is None:
        q_prequant = torch.empty((M, Q_DIM), dtype=torch.float32, device=latent.device)
    if fp4_format != "mx":
        if q_prequant is not None:
            _require(q_prequant, "q_prequant", (torch.float32,), (M, Q_DIM))
        _check(lib().iq_prepare_q_ex(_ptr(latent), M, _ptr(wq), _ptr(wq_sf), _ptr(positions),
                                     FP4_FORMATS[fp4_format], _ptr(q_fp4), _ptr(q_sf), _ptr(q_prequant),
                                     _ptr(workspace), workspace.numel(), _stream(stream)), "iq_prepare_q_ex")
        return (q_fp4, q_sf, q_prequant) if q_prequant is not None else (q_fp4, q_sf)
    if q_prequant is not None:
        _require(q_prequant, "q_prequant", (torch.float32,), (M, Q_DIM))
        _check(lib().iq_prepare_q_debug(_ptr(latent), M, _ptr(wq), _ptr(wq_sf), _ptr(positions), _ptr(q_fp4),
                                        _ptr(q_sf), _ptr(q_prequant), _ptr(workspace), workspace.numel(),
                                        _stream(stream)), "iq_prepare_q_debug")
        return q_fp4, q_sf, q_prequant
    _check(lib().iq_prepare_q(_ptr(latent), M, _ptr(wq), _ptr(wq_sf), _ptr(positions), _ptr(q_fp4), _ptr(q_sf),
                              _ptr(workspace), workspace.numel(), _stream(stream)), "iq_prepare_q")
    return q_fp4, q_sf


def _require_host_side(t: torch.Tensor, name: str, dtypes, shape):
    """A page-locked CPU tensor (or a CUDA tensor) of the given dtype and shape."""
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be in page-locked host memory (tensor.pin_memory()) or on the GPU")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def prepare_q_host_workspace_bytes(M: int, fp4_format: str = "mx") -> int:
    return int(lib().iq_prepare_q_host_workspace(M, FP4_FORMATS[fp4_format]))


def prepare_q_host(latent: torch.Tensor, wq: torch.Tensor, wq_sf: torch.Tensor, positions: torch.Tensor, *,
                   q_fp4: torch.Tensor | None = None, q_sf: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None, fp4_format: str = "mx", stream=None):
    """Indexer-Q preparation on host-resident tokens (iq_prepare_q_host):
    latent [M, 1536] bf16 and positions [M] int32 in page-locked host memory;
    returns (q_fp4 uint8 [M, 4096], q_sf uint8 [M, 256] or [M, 512]) in
    page-locked host memory, complete once `stream` reaches the point after
    this call.  W and its scales are on the GPU."""
    M = latent.shape[0]
    if fp4_format not in FP4_FORMATS:
        raise ValueError(f"fp4_format must be one of {sorted(FP4_FORMATS)}")
    _require_host_side(latent, "latent", (torch.bfloat16,), (M, LATENT_DIM))
    _require_host_side(positions, "positions", (torch.int32,), (M,))
    _require(wq, "wq", _U8, (Q_DIM, LATENT_DIM))
    _require(wq_sf, "wq_sf", (torch.uint8,), (N_HEADS, LATENT_DIM // 128))
    sf_cols = Q_DIM // 16 if fp4_format == "nv" else Q_DIM // 32
    if q_fp4 is None:
        q_fp4 = torch.empty((M, Q_DIM // 2), dtype=torch.uint8).pin_memory()
    if q_sf is None:
        q_sf = torch.empty((M, sf_cols), dtype=torch.uint8).pin_memory()
    _require_host_side(q_fp4, "q_fp4", (torch.uint8,), (M, Q_DIM // 2))
    _require_host_side(q_sf, "q_sf", (torch.uint8,), (M, sf_cols))
    if workspace is None:
        workspace = torch.empty(max(prepare_q_host_workspace_bytes(M, fp4_format), 1), dtype=torch.uint8,
                                device=wq.device)
    _require(workspace, "workspace", (torch.uint8,))
    _check(lib().iq_prepare_q_host(_ptr(latent), M, _ptr(wq), _ptr(wq_sf), _ptr(positions),
                                   FP4_FORMATS[fp4_format], _ptr(q_fp4), _ptr(q_sf), _ptr(workspace),
                                   workspace.numel(), _stream(stream)), "iq_prepare_q_host")
    return q_fp4, q_sf


def set_host_chunk_rows(rows: int) -> int:
    """Rows per chunk of prepare_q_host (a multiple of 256); returns the
    previous value."""
    return int(lib().iq_set_host_chunk_rows(int(rows)))


def host_chunk_rows() -> int:
    return int(lib().iq_host_chunk_rows())


def gemm_rope_hadamard_fp4(xq: torch.Tensor, x_scales: torch.Tensor, wq: torch.Tensor, wq_sf: torch.Tensor,
                           positions: torch.Tensor, *, q_fp4: torch.Tensor | None = None,
                           q_sf: torch.Tensor | None = None, q_prequant: torch.Tensor | None = None, stream=None):
    """Second stage alone on an FP8 latent [M, 1536] and its packed scales
    [3, align4(M)]."""
    M = xq.shape[0]
    _require(xq, "xq", _U8, (M, LATENT_DIM))
    _require(x_scales, "x_scales", (torch.int32,), (3, (M + 3) // 4 * 4))
    _require(wq, "wq", _U8, (Q_DIM, LATENT_DIM))
    _require(wq_sf, "wq_sf", (torch.uint8,), (N_HEADS, LATENT_DIM // 128))
    _require(positions, "positions", (torch.int32,), (M,))
    q_fp4, q_sf = _prepare_out(M, xq.device, q_fp4, q_sf)
    if q_prequant is not None:
        _require(q_prequant, "q_prequant", (torch.float32,), (M, Q_DIM))
    _check(lib().iq_gemm_rope_hadamard_fp4(_ptr(xq), _ptr(x_scales), M, _ptr(wq), _ptr(wq_sf), _ptr(positions),
                                           _ptr(q_fp4), _ptr(q_sf), _ptr(q_prequant), _stream(stream)),
           "iq_gemm_rope_hadamard_fp4")
    return q_fp4, q_sf


def device_status(reset: bool = False) -> int:
    """Device status word (bits of waits that gave up); synchronizes."""
    v = ctypes.c_uint32(0)
    code = lib().iq_device_status(ctypes.byref(v), 1 if reset else 0)
    if code not in (0, -7):
        raise IQError(code, "iq_device_status")
    return int(v.value)


def set_gemm_tiling(tile_n: int = 0, order: int = 0) -> None:
    """Tuning override of the CTA-pair kernel's tiling (include/iq.h,
    iq_set_gemm_tiling): tile_n 128 or 256, order 1 feature-major, 2
    token-major or 3 interleaved; 0 restores the default."""
    lib().iq_set_gemm_tiling(int(tile_n), int(order))


def set_quant_fusion(on: bool) -> bool:
    """The quantizer fused into the CTA-pair kernel (include/iq.h,
    iq_set_quant_fusion); returns the previous setting."""
    return bool(lib().iq_set_quant_fusion(1 if on else 0))


def debug_delay_quant_ns(ns: int) -> None:
    """Diagnostics: delay of the fused quantizer's signals (iq_debug_delay_quant_ns)."""
    lib().iq_debug_delay_quant_ns(int(ns))


def set_wait_timeout_ns(ns: int) -> None:
    lib().iq_set_wait_timeout_ns(int(ns))


def set_small_m_threshold(max_tokens: int) -> int:
    """Largest M routed to the small-M (swapped-operand) kernel, clamped to
    [0, 64]; returns the previous value."""
    return int(lib().iq_set_small_m_threshold(int(max_tokens)))


def small_m_threshold() -> int:
    return int(lib().iq_small_m_threshold())


def indexer_logits(q_fp4: torch.Tensor, q_sf: torch.Tensor, k_fp4: torch.Tensor, k_sf: torch.Tensor,
                   weights: torch.Tensor, lengths: torch.Tensor, *, logits: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """Indexer scores (include/iq.h, iq_indexer_logits): q_fp4 uint8 [M, 4096],
    q_sf uint8 [M, 256], k_fp4 uint8 [N, 64], k_sf uint8 [N, 4], weights
    float32 [M, 64], lengths int32 [M] -> logits float32 [M, N] (row stride may
    exceed N); entries at s >= lengths[t] are left as they were."""
    M, N = q_fp4.shape[0], k_fp4.shape[0]
    _require(q_fp4, "q_fp4", (torch.uint8,), (M, Q_DIM // 2))
    _require(q_sf, "q_sf", (torch.uint8,), (M, Q_DIM // 32))
    _require(k_fp4, "k_fp4", (torch.uint8,), (N, HEAD_DIM // 2))
    _require(k_sf, "k_sf", (torch.uint8,), (N, HEAD_DIM // 32))
    _require(weights, "weights", (torch.float32,), (M, N_HEADS))
    _require(lengths, "lengths", (torch.int32,), (M,))
    if logits is None:
        logits = torch.empty((M, N), dtype=torch.float32, device=q_fp4.device)
    if logits.dim() != 2 or logits.shape[0] != M or logits.shape[1] < N or logits.stride(1) != 1:
        raise ValueError("logits must be float32 [M, >= N] with unit column stride")
    _require(logits, "logits", (torch.float32,), contiguous=False)
    _check(lib().iq_indexer_logits(_ptr(q_fp4), _ptr(q_sf), M, _ptr(k_fp4), _ptr(k_sf), N, _ptr(weights),
                                   _ptr(lengths), _ptr(logits), logits.stride(0), _stream(stream)),
           "iq_indexer_logits")
    return logits


def indexer_topk(logits: torch.Tensor, lengths: torch.Tensor, k: int, *, N: int | None = None,
                 indices: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Top-k key selection per query row (include/iq.h, iq_indexer_topk):
    int32 [M, k] ascending indices, -1 padded.  N defaults to logits.shape[1]."""
    M = logits.shape[0]
    N = logits.shape[1] if N is None else N
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be a 2-D tensor with unit column stride")
    _require(logits, "logits", (torch.float32,), contiguous=False)
    _require(lengths, "lengths", (torch.int32,), (M,))
    if indices is None:
        indices = torch.empty((M, k), dtype=torch.int32, device=logits.device)
    _require(indices, "indices", (torch.int32,), (M, k))
    _check(lib().iq_indexer_topk(_ptr(logits), logits.stride(0), M, N, _ptr(lengths), int(k), _ptr(indices),
                                 _stream(stream)), "iq_indexer_topk")
    return indices
