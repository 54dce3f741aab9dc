"""GPU parity of the FP4 output variants (include/iq.h, iq_prepare_q_ex)
against the CPU oracle, on both GEMM routes: the OCP MX floor rule and the
NVFP4-style 1x16 blocks with E4M3 scales."""

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


def _dev(x, pos, wq, wsf):
    lat = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return lat, torch.from_numpy(wq).cuda(), torch.from_numpy(wsf).cuda(), torch.from_numpy(pos).cuda()


def _run(x, wq, wsf, pos, fmt):
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    q, sf, z = _iq().prepare_q(lat, w, ws, p, debug=True, fp4_format=fmt)
    torch.cuda.synchronize()
    return q.cpu().numpy(), sf.cpu().numpy(), z.cpu().numpy()


@pytest.mark.parametrize("fmt", ["mx_ocp", "nv"])
@pytest.mark.parametrize("M", [1, 16, 64, 100, 300, 1024])
def test_variant_matches_oracle(cuda_device, fmt, M):
    x, wq, wsf, pos = W.chain_workload(M, seed=6000 + M, outlier_p=0.005, outlier_scale=100.0)
    q, sf, z = _run(x, wq, wsf, pos, fmt)
    oq, osf, oz = O.prepare_q(x, wq, wsf, pos, fmt)
    check_prequant(z, oz)
    stats = check_fp4(q, sf, oq, osf, oz, fmt=fmt)
    assert stats["equal_fraction"] >= 0.9999
    assert _iq().device_status() == 0


@pytest.mark.parametrize("fmt", ["mx_ocp", "nv"])
def test_variant_prefill_4632(cuda_device, fmt):
    x, wq, wsf, pos = W.prefill_chain(4632)
    q, sf, z = _run(x, wq, wsf, pos, fmt)
    oq, osf, oz = O.prepare_q(x, wq, wsf, pos, fmt)
    check_prequant(z, oz)
    print(fmt, check_fp4(q, sf, oq, osf, oz, fmt=fmt))


@pytest.mark.parametrize("M", [9, 200])
def test_variant_zero_latent(cuda_device, M):
    x, wq, wsf, pos = W.chain_workload(M, seed=1, outlier_p=0.0, outlier_scale=1.0)
    x = np.zeros_like(x)
    for fmt, floor_byte in (("mx_ocp", 111), ("nv", 1)):
        q, sf, z = _run(x, wq, wsf, pos, fmt)
        assert np.all((q & 0x77) == 0) and np.all(sf == floor_byte), fmt
        check_fp4(q, sf, *O.prepare_q(x, wq, wsf, pos, fmt), fmt=fmt)


@pytest.mark.parametrize("M", [7, 300])
def test_default_format_through_ex_equals_prepare_q(cuda_device, M):
    iq = _iq()
    L = iq.lib()
    x, wq, wsf, pos = W.chain_workload(M, seed=77, outlier_p=0.001, outlier_scale=50.0)
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    q1, s1 = iq.prepare_q(lat, w, ws, p)
    q2 = torch.empty_like(q1)
    s2 = torch.empty_like(s1)
    work = torch.empty(iq.prepare_q_workspace_bytes(M), dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert L.iq_prepare_q_ex(lat.data_ptr(), M, w.data_ptr(), ws.data_ptr(), p.data_ptr(), 0, q2.data_ptr(),
                             s2.data_ptr(), None, work.data_ptr(), work.numel(), st) == 0
    torch.cuda.synchronize()
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
