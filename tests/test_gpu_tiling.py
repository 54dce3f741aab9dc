"""The CTA-pair kernel's tilings: one head (128 features) or two heads (256)
per pair tile; feature-major, token-major or interleaved tile order.  Every
setting computes each output with the same sums in the same order, so all of
them must give the same bytes, and the default route must match the oracle at
the mid-size token counts.  The tilings are exercised with the quantizer as a
separate launch (the fused route always takes two-head tiles in the
interleaved order)."""

import contextlib

import numpy as np
import pytest
import torch

from oracle import iq_oracle as O
from fp4_fp8_quant_gb300 import workloads as W
from tests.parity import check_fp4, check_prequant

pytestmark = pytest.mark.gpu


def _iq():
    from fp4_fp8_quant_gb300 import iq
    return iq


@contextlib.contextmanager
def _tiling(tile_n, order):
    iq = _iq()
    iq.set_gemm_tiling(tile_n, order)
    prev = iq.set_quant_fusion(False)
    route = iq.set_small_m_threshold(0)   # every M on the CTA-pair kernel
    try:
        yield
    finally:
        iq.set_gemm_tiling(0, 0)
        iq.set_quant_fusion(prev)
        iq.set_small_m_threshold(route)


def _dev(x, pos, wq, wsf):
    lat = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return lat, torch.from_numpy(wq).cuda(), torch.from_numpy(wsf).cuda(), torch.from_numpy(pos).cuda()


@pytest.mark.parametrize("M", [65, 100, 128, 129, 200, 256, 512, 1024])
def test_mid_size_token_counts_match_oracle(cuda_device, M):
    x, wq, wsf, pos = W.sweep_chain(M, seed=700 + M)
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    q, sf, z = _iq().prepare_q(lat, w, ws, p, debug=True)
    torch.cuda.synchronize()
    oq, osf, oz = O.prepare_q(x, wq, wsf, pos)
    check_prequant(z.cpu().numpy(), oz)
    check_fp4(q.cpu().numpy(), sf.cpu().numpy(), oq, osf, oz)
    assert _iq().device_status() == 0


@pytest.mark.parametrize("M", [100, 777, 2048 + 37])
@pytest.mark.parametrize("fmt", ["mx", "nv"])
def test_every_tiling_gives_the_same_bytes(cuda_device, M, fmt):
    iq = _iq()
    x, wq, wsf, pos = W.sweep_chain(M, seed=800 + M)
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    outs = {}
    for tile_n in (128, 256):
        for order in (1, 2, 3):
            with _tiling(tile_n, order):
                outs[(tile_n, order)] = iq.prepare_q(lat, w, ws, p, debug=True, fp4_format=fmt)
    torch.cuda.synchronize()
    ref = outs[(256, 1)]
    for key, out in outs.items():
        for a, b in zip(out, ref):
            assert torch.equal(a, b), (key, fmt)
    oq, osf, oz = O.prepare_q(x, wq, wsf, pos, fmt)
    check_prequant(ref[2].cpu().numpy(), oz)
    check_fp4(ref[0].cpu().numpy(), ref[1].cpu().numpy(), oq, osf, oz, fmt=fmt)
    assert iq.device_status() == 0


def test_token_major_order_at_a_sweep_size(cuda_device):
    """16384 tokens take the token-major order by default; sampled rows
    against the oracle, all rows against the feature-major order."""
    iq = _iq()
    M = 16384
    x, wq, wsf, pos = W.sweep_chain(M)
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    q, sf = iq.prepare_q(lat, w, ws, p)
    with _tiling(256, 1):
        q1, sf1 = iq.prepare_q(lat, w, ws, p)
    torch.cuda.synchronize()
    assert torch.equal(q, q1) and torch.equal(sf, sf1)
    rows = np.unique(np.concatenate([np.random.default_rng(5).choice(M, 48, replace=False), [0, 255, 256, M - 1]]))
    oq, osf, oz = O.prequant_q_rows(x, wq, wsf, pos, rows)
    check_fp4(q.cpu().numpy()[rows], sf.cpu().numpy()[rows], oq, osf, oz)
    assert iq.device_status() == 0
