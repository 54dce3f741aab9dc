"""GPU parity of the small-M route (the swapped-operand kernel that
iq_prepare_q runs for 1 <= M <= 128 tokens: 64 token columns up to 64
tokens, 128 above) against the CPU oracle, and its agreement with the CTA-pair
kernel at the same token counts.

Both routes compute the same operation; their float32 sums are formed in a
different order (the small-M kernel splits K in two halves and adds the
halves' sums), so they are compared with the oracle under the rules of
tests/parity.py, not with each other byte for byte.
"""

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
def _route(threshold):
    iq = _iq()
    old = iq.set_small_m_threshold(threshold)
    try:
        yield
    finally:
        iq.set_small_m_threshold(old)


def _dev(x, pos, wq, wsf):
    lat = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return lat, torch.from_numpy(wq).cuda(), torch.from_numpy(wsf).cuda(), torch.from_numpy(pos).cuda()


def _run(x, wq, wsf, pos):
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    q, sf, z = _iq().prepare_q(lat, w, ws, p, debug=True)
    torch.cuda.synchronize()
    return q.cpu().numpy(), sf.cpu().numpy(), z.cpu().numpy()


@pytest.mark.parametrize("M", [1, 2, 3, 7, 8, 9, 17, 31, 32, 33, 48, 63, 64, 65, 66, 77, 96, 100, 127, 128])
def test_small_m_route_matches_oracle(cuda_device, M):
    x, wq, wsf, pos = W.chain_workload(M, seed=500 + M, outlier_p=0.005, outlier_scale=100.0)
    with _route(128):
        q, sf, z = _run(x, wq, wsf, pos)
    oq, osf, oz = O.prepare_q(x, wq, wsf, pos)
    check_prequant(z, oz)
    check_fp4(q, sf, oq, osf, oz)
    assert _iq().device_status() == 0


@pytest.mark.parametrize("M", [1, 8, 32, 64, 96, 128])
def test_small_m_decode_workload(cuda_device, M):
    """The decode inputs: N(0,1) latent, random positions up to 163840."""
    x, wq, wsf, pos = W.decode_chain(M)
    with _route(128):
        q, sf, z = _run(x, wq, wsf, pos)
    oq, osf, oz = O.prepare_q(x, wq, wsf, pos)
    check_prequant(z, oz)
    stats = check_fp4(q, sf, oq, osf, oz)
    assert stats["equal_fraction"] >= 0.9999


@pytest.mark.parametrize("M", [1, 5, 64, 65, 128])
def test_both_routes_agree_with_the_oracle_and_each_other(cuda_device, M):
    x, wq, wsf, pos = W.chain_workload(M, seed=900 + M, outlier_p=0.001, outlier_scale=50.0)
    oq, osf, oz = O.prepare_q(x, wq, wsf, pos)
    outs = []
    for threshold in (0, 128):
        with _route(threshold):
            q, sf, z = _run(x, wq, wsf, pos)
        check_prequant(z, oz)
        check_fp4(q, sf, oq, osf, oz)
        outs.append((q, sf, z))
    # The two float32 results differ by rounding only.
    rms = np.sqrt(np.mean(oz ** 2, axis=1, keepdims=True))
    assert np.all(np.abs(outs[0][2] - outs[1][2]) <= 2e-4 * rms)
    assert (outs[0][1] == outs[1][1]).mean() > 0.999


def test_small_m_zero_latent_and_extreme_positions(cuda_device):
    M = 12
    x, wq, wsf, pos = W.chain_workload(M, seed=77, outlier_p=0.0, outlier_scale=1.0)
    x[3] = 0                                   # one all-zero token
    pos = np.array([0, 1, 163839, 2 ** 23, 5, 65535, 100000, 7, 8, 9, 10, 163838], dtype=np.int32)
    with _route(128):
        q, sf, z = _run(x, wq, wsf, pos)
    oq, osf, oz = O.prepare_q(x, wq, wsf, pos)
    check_prequant(z, oz)
    check_fp4(q, sf, oq, osf, oz)
    assert np.all((q[3] & 0x77) == 0) and np.all(sf[3] == 112)


@pytest.mark.parametrize("M", [24, 100])
def test_small_m_graph_replay_and_static_entry(cuda_device, M):
    """A captured small-M call replays to the eager result; the allocation-free
    entry point takes the same route."""
    iq = _iq()
    L = iq.lib()
    x, wq, wsf, pos = W.decode_chain(M)
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    with _route(128):
        work = torch.empty(iq.prepare_q_workspace_bytes(M), dtype=torch.uint8, device="cuda")
        q = torch.empty((M, 4096), dtype=torch.uint8, device="cuda")
        s = torch.empty((M, 256), dtype=torch.uint8, device="cuda")
        iq.prepare_q(lat, w, ws, p, q_fp4=q, q_sf=s, workspace=work)
        torch.cuda.synchronize()
        qe, se = q.clone(), s.clone()
        q.zero_()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                iq.prepare_q(lat, w, ws, p, q_fp4=q, q_sf=s, workspace=work)
        for _ in range(5):
            g.replay()
        torch.cuda.synchronize()
        assert torch.equal(q, qe) and torch.equal(s, se)
        q2 = torch.zeros_like(q)
        s2 = torch.zeros_like(s)
        st = torch.cuda.current_stream().cuda_stream
        assert L.iq_prepare_q_static(lat.data_ptr(), M, w.data_ptr(), ws.data_ptr(), p.data_ptr(), q2.data_ptr(),
                                     s2.data_ptr(), st) == 0
        torch.cuda.synchronize()
        assert torch.equal(q2, qe) and torch.equal(s2, se)
    assert iq.device_status() == 0
