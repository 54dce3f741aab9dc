"""iq_prepare_q_static: indexer-Q preparation that allocates nothing.

Some callers cannot hand the library a workspace: a plugin inside a host
program that owns all device memory and exposes no allocator to it, or a
latency-bound loop that must not call cudaMalloc (which may synchronize the
whole device).  For them the library keeps the FP8 latent in a scratch array
of its own, sized for at most IQ_STATIC_MAX_TOKENS tokens.

These tests call the entry point through the C ABI twice in a row with
different inputs (the second call runs on whatever the first left in the
shared scratch) and check each result against iq_prepare_q, the entry point
with a caller workspace.  Both run the same kernels on the same data, so the
outputs must agree byte for byte, which is within every tolerance the parity
tests allow.  The file name sorts last so that a run stopping at the first
failure has already run every other test.
"""

import numpy as np
import pytest
import torch

from fp4_fp8_quant_gb300 import workloads as W

pytestmark = pytest.mark.gpu

IQ_STATIC_MAX_TOKENS = 2048
IQ_ERR_WORKSPACE = -6


def _inputs(M, seed):
    x, wq, wsf, pos = W.chain_workload(M, seed=seed, outlier_p=0.005, outlier_scale=100.0)
    lat = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    return lat, torch.from_numpy(wq).cuda(), torch.from_numpy(wsf).cuda(), torch.from_numpy(pos).cuda()


def _call_static(L, lat, w, ws, p, q, s):
    st = torch.cuda.current_stream().cuda_stream
    return L.iq_prepare_q_static(lat.data_ptr(), lat.shape[0], w.data_ptr(), ws.data_ptr(), p.data_ptr(),
                                 q.data_ptr(), s.data_ptr(), st)


def test_static_scratch_matches_workspace_entry_point_twice_in_a_row(cuda_device):
    from fp4_fp8_quant_gb300 import iq
    L = iq.lib()
    for M, seed in ((300, 41), (37, 42), (IQ_STATIC_MAX_TOKENS, 43)):
        lat, w, ws, p = _inputs(M, seed)
        q = torch.full((M, 4096), 0xAB, dtype=torch.uint8, device="cuda")
        s = torch.full((M, 256), 0xAB, dtype=torch.uint8, device="cuda")
        assert _call_static(L, lat, w, ws, p, q, s) == 0
        q_ref, s_ref = iq.prepare_q(lat, w, ws, p)
        torch.cuda.synchronize()
        assert torch.equal(q, q_ref), f"FP4 codes differ from iq_prepare_q at M={M}"
        assert torch.equal(s, s_ref), f"FP4 scales differ from iq_prepare_q at M={M}"
    assert iq.device_status() == 0


def test_static_scratch_rejects_too_many_tokens(cuda_device):
    from fp4_fp8_quant_gb300 import iq
    L = iq.lib()
    M = IQ_STATIC_MAX_TOKENS + 1
    lat, w, ws, p = _inputs(M, 44)
    q = torch.empty((M, 4096), dtype=torch.uint8, device="cuda")
    s = torch.empty((M, 256), dtype=torch.uint8, device="cuda")
    assert _call_static(L, lat, w, ws, p, q, s) == IQ_ERR_WORKSPACE
    empty = torch.empty((0, 1536), dtype=torch.bfloat16, device="cuda")
    assert _call_static(L, empty, w, ws, p, q, s) == 0
    torch.cuda.synchronize()
