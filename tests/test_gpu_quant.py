"""GPU parity of the FP8 1x128 quantizer (iq_fp8_quant_1x128_ue8m0) against
the CPU oracle: codes and packed scale words bit-exact."""

import numpy as np
import pytest
import torch

from oracle import iq_oracle as O
from fp4_fp8_quant_gb300 import workloads as W
from tests.parity import check_fp8

pytestmark = pytest.mark.gpu


def _iq():
    from fp4_fp8_quant_gb300 import iq
    return iq


def _to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _run(bits):
    iq = _iq()
    y, s = iq.fp8_quant_1x128_ue8m0(_to_dev(bits))
    torch.cuda.synchronize()
    return y.cpu().numpy(), s.cpu().numpy()


def test_quantizer_full_size_blocks_workload(cuda_device):
    """[4632, 7168] with 1% x1e3 blocks, 1% zero blocks, 1% tiny blocks."""
    bits = W.quant_blocks_input(4632, 7168, seed=1)
    y, s = _run(bits)
    oc, ow = O.fp8_quant_1x128_ue8m0(bits)
    check_fp8(y, s, oc, ow)
    sb = (ow.view(np.uint32)[:, :4632, None] >> np.array([0, 8, 16, 24], dtype=np.uint32)) & 0xFF
    assert (sb == 105).sum() > 1000          # floored blocks are present


@pytest.mark.parametrize("M,K", [(1, 128), (3, 384), (4, 1536), (5, 640), (7, 2048), (129, 7168), (16, 1536),
                                 (1000, 896)])
def test_quantizer_shapes_and_tails(cuda_device, M, K):
    bits = W.quant_blocks_input(M, K, seed=M * 31 + K, p_large=0.05, p_zero=0.05, p_tiny=0.05)
    y, s = _run(bits)
    check_fp8(y, s, *O.fp8_quant_1x128_ue8m0(bits))


def test_quantizer_every_bf16_pattern(cuda_device):
    """All finite BF16 values, sorted by magnitude into 1x128 blocks (so that
    each value is quantized next to values of its own size) and, separately,
    in a seeded shuffle (so that small values meet large block scales)."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = O.bf16_bits_to_f64(allbits)
    fin = allbits[np.isfinite(v)]
    order = np.argsort(np.abs(O.bf16_bits_to_f64(fin)), kind="stable")
    pad = (-len(fin)) % 128
    for arr in (fin[order], np.random.default_rng(0).permutation(fin)):
        arr = np.concatenate([arr, np.zeros(pad, np.uint16)]).reshape(-1, 128)
        y, s = _run(arr)
        check_fp8(y, s, *O.fp8_quant_1x128_ue8m0(arr))


def test_quantizer_signed_zero(cuda_device):
    bits = np.zeros((2, 128), np.uint16)
    bits[0, :4] = [0x8000, 0x3F80, 0xB380, 0x0000]   # -0, 1.0, -6e-8 (rounds to -0), +0
    y, s = _run(bits)
    assert y[0, 0] == 0x80 and y[0, 2] == 0x80 and y[0, 3] == 0x00
    check_fp8(y, s, *O.fp8_quant_1x128_ue8m0(bits))


def test_quantizer_strided_rows(cuda_device):
    iq = _iq()
    M, K = 37, 1024
    bits = W.quant_blocks_input(M, K, seed=5)
    big = torch.zeros((M, K + 64), dtype=torch.bfloat16, device="cuda")
    big[:, :K] = _to_dev(bits)
    yb = torch.full((M, K + 32), 0x5A, dtype=torch.uint8, device="cuda")
    y, s = iq.fp8_quant_1x128_ue8m0(big[:, :K], y=yb[:, :K])
    torch.cuda.synchronize()
    check_fp8(y.cpu().numpy(), s.cpu().numpy(), *O.fp8_quant_1x128_ue8m0(bits))
    assert torch.all(yb[:, K:] == 0x5A)       # padding columns untouched


def test_quantizer_empty_and_errors(cuda_device):
    iq = _iq()
    L = iq.lib()
    x = torch.zeros((8, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((8, 256), dtype=torch.uint8, device="cuda")
    s = torch.zeros((1, 8), dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert L.iq_fp8_quant_1x128_ue8m0(x.data_ptr(), 0, 256, 256, y.data_ptr(), 256, s.data_ptr(), st) == 0
    assert L.iq_fp8_quant_1x128_ue8m0(x.data_ptr(), 8, 200, 256, y.data_ptr(), 256, s.data_ptr(), st) == -3
    assert L.iq_fp8_quant_1x128_ue8m0(x.data_ptr() + 2, 8, 128, 256, y.data_ptr(), 256, s.data_ptr(), st) == -2
    assert L.iq_fp8_quant_1x128_ue8m0(x.data_ptr(), 8, 128, 136, y.data_ptr(), 256, s.data_ptr(), st) == 0
    assert L.iq_fp8_quant_1x128_ue8m0(x.data_ptr(), 8, 128, 132, y.data_ptr(), 256, s.data_ptr(), st) == -2
    assert L.iq_fp8_quant_1x128_ue8m0(None, 8, 128, 256, y.data_ptr(), 256, s.data_ptr(), st) == -1
    assert L.iq_fp8_quant_1x128_ue8m0(x.data_ptr(), -1, 128, 256, y.data_ptr(), 256, s.data_ptr(), st) == -1
    torch.cuda.synchronize()


@pytest.mark.parametrize("M", [16384, 65536])
def test_quantizer_long_prefill_sweep_sizes(cuda_device, M):
    """The sweep's quantizer leg, BF16 [M, 7168] with 0.5% of elements x100
    (up to 114,688 warps and 470 M elements per launch).  Rows are
    independent: a seeded sample of rows (the first and last, and rows around
    the 4-row scale-word groups) is compared with the oracle bit for bit; every
    row is checked on the device against the scale rule and the E4M3 rounding
    bound."""
    K = 7168
    iq = _iq()
    x = torch.empty((M, K), dtype=torch.int16, device="cuda")
    for b in range((M + W.SWEEP_ROW_BLOCK - 1) // W.SWEEP_ROW_BLOCK):
        blk = W.sweep_quant_block(M, K, b)
        r0 = b * W.SWEEP_ROW_BLOCK
        x[r0:r0 + blk.shape[0]] = torch.from_numpy(blk.view(np.int16)).cuda()
    xb = x.view(torch.bfloat16)
    y, s = iq.fp8_quant_1x128_ue8m0(xb)
    torch.cuda.synchronize()

    rng = np.random.default_rng(M + 17)
    rows = np.unique(np.concatenate([rng.choice(M, 60, replace=False), [0, 1, 2, 3, 4, M - 5, M - 1]]))
    bits = W.sweep_quant_rows(M, K, rows)
    assert np.array_equal(bits, x[torch.from_numpy(rows).cuda()].cpu().numpy().view(np.uint16))
    oc, osb = O.quantize_fp8_1x128(O.bf16_bits_to_f64(bits))
    yc = y[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert np.array_equal(yc, oc), f"{int((yc != oc).sum())} FP8 code mismatches on sampled rows"
    words = s.cpu().numpy().view(np.uint32)
    assert words.shape == (K // 512, M)
    gsb = (words[:, rows].T[:, :, None] >> np.array([0, 8, 16, 24], np.uint32)) & 0xFF
    assert np.array_equal(gsb.reshape(len(rows), -1)[:, :K // 128], osb)

    # every row: the scale byte is the ceil rule on the floored amax, and each
    # decoded code lies within half an E4M3 step of x * 2^-e
    xf = xb.float().view(M, K // 128, 128)
    e = (words[:, None, :] >> np.array([0, 8, 16, 24], np.uint32)[None, :, None]) & 0xFF
    e = torch.from_numpy(e.reshape(-1, M).T[:, :K // 128].astype(np.int32) - 127).cuda()
    amax = xf.abs().amax(dim=2).clamp_min(1e-4)
    two_e = torch.ldexp(torch.ones_like(amax), e)
    assert bool(((448.0 * two_e >= amax) & (224.0 * two_e < amax)).all()), "scale exponent breaks the ceil rule"
    u = xf / two_e[..., None]
    dec = y.view(torch.float8_e4m3fn).float().view(M, K // 128, 128)
    _, ex = torch.frexp(u.abs())
    half_step = torch.ldexp(torch.ones_like(u), torch.clamp(ex - 1, min=-6) - 4)
    assert bool(((dec - u).abs() <= half_step).all()), "a code lies more than half a step from x * 2^-e"
