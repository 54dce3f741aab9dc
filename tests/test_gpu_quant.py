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
