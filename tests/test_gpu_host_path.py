"""The host-buffer entry (iq_prepare_q_host): token rows and results in
page-locked host memory, processed in row chunks whose transfers overlap the
computation.

Its results are checked against the CPU oracle at sizes where chunks of 256
rows leave ragged tails on both GEMM routes (a last chunk of more than 128
rows takes the CTA-pair kernel, one of at most 128 the small-M kernel), and byte
for byte against the device-buffer entry at the 4,632-token prefill size,
where every chunk takes the CTA-pair kernel: a row's arithmetic does not
depend on the chunk or tile it falls in.
"""

import contextlib

import numpy as np
import pytest
import torch

from oracle import iq_oracle as O
from fp4_fp8_quant_gb300 import workloads as W
from tests.parity import check_fp4

pytestmark = pytest.mark.gpu


def _iq():
    from fp4_fp8_quant_gb300 import iq
    return iq


@contextlib.contextmanager
def _chunk_rows(rows):
    iq = _iq()
    old = iq.set_host_chunk_rows(rows)
    try:
        yield
    finally:
        iq.set_host_chunk_rows(old)


def _host_inputs(x, pos):
    lat = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).pin_memory()
    return lat, torch.from_numpy(np.ascontiguousarray(pos)).pin_memory()


def _weights(wq, wsf):
    return torch.from_numpy(wq).cuda(), torch.from_numpy(wsf).cuda()


def _run_host(x, wq, wsf, pos, fmt="mx"):
    lat, p = _host_inputs(x, pos)
    w, ws = _weights(wq, wsf)
    q, sf = _iq().prepare_q_host(lat, w, ws, p, fp4_format=fmt)
    torch.cuda.current_stream().synchronize()
    assert not q.is_cuda and q.is_pinned()
    return q.numpy(), sf.numpy()


@pytest.mark.parametrize("M,rows", [(16, 1024), (300, 256), (600, 256), (1000, 512)])
def test_host_entry_matches_oracle(cuda_device, M, rows):
    x, wq, wsf, pos = W.chain_workload(M, seed=1200 + M, outlier_p=0.005, outlier_scale=100.0)
    with _chunk_rows(rows):
        q, sf = _run_host(x, wq, wsf, pos)
    oq, osf, oz = O.prepare_q(x, wq, wsf, pos)
    stats = check_fp4(q, sf, oq, osf, oz)
    assert stats["equal_fraction"] >= 0.9999
    assert _iq().device_status() == 0


@pytest.mark.parametrize("fmt", ["mx_ocp", "nv"])
def test_host_entry_fp4_variants(cuda_device, fmt):
    M = 300
    x, wq, wsf, pos = W.chain_workload(M, seed=1300, outlier_p=0.005, outlier_scale=100.0)
    with _chunk_rows(256):
        q, sf = _run_host(x, wq, wsf, pos, fmt)
    oq, osf, oz = O.prepare_q(x, wq, wsf, pos, fmt)
    check_fp4(q, sf, oq, osf, oz, fmt=fmt)


@pytest.mark.parametrize("rows", [1024, 1280, 2048, 4864])
def test_host_entry_equals_device_entry_at_prefill_size(cuda_device, rows):
    """Chunk sizes whose last chunk (536, 792, 536 and 4632 rows) also takes
    the CTA-pair kernel; a multiple of 256 that divides 4608 would leave a
    24-row chunk to the small-M kernel, whose float32 sums are ordered
    differently (that route is checked against the oracle above)."""
    M = 4632
    x, wq, wsf, pos = W.prefill_chain(M)
    w, ws = _weights(wq, wsf)
    lat_d = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    qd, sfd = _iq().prepare_q(lat_d, w, ws, torch.from_numpy(pos).cuda())
    with _chunk_rows(rows):
        qh, sfh = _run_host(x, wq, wsf, pos)
    assert np.array_equal(qh, qd.cpu().numpy())
    assert np.array_equal(sfh, sfd.cpu().numpy())


def test_host_entry_accepts_device_buffers(cuda_device):
    """Device-resident inputs and outputs are accepted (the copies are then
    device to device) and give the device entry's bytes."""
    M = 700
    x, wq, wsf, pos = W.decode_chain(M)
    w, ws = _weights(wq, wsf)
    lat_d = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    p_d = torch.from_numpy(pos).cuda()
    qd, sfd = _iq().prepare_q(lat_d, w, ws, p_d)
    q2 = torch.empty_like(qd)
    sf2 = torch.empty_like(sfd)
    with _chunk_rows(256):
        _iq().prepare_q_host(lat_d, w, ws, p_d, q_fp4=q2, q_sf=sf2)
    torch.cuda.synchronize()
    assert torch.equal(q2, qd) and torch.equal(sf2, sfd)


def test_host_entry_back_to_back_calls_reuse_the_workspace(cuda_device):
    """Three calls on one stream and one workspace: each call's results are
    those of its own inputs."""
    iq = _iq()
    M = 520
    cases = [W.chain_workload(M, seed=1400 + i, outlier_p=0.001, outlier_scale=50.0) for i in range(3)]
    w, ws = _weights(cases[0][1], cases[0][2])   # W does not depend on the seed of the tokens
    for (_, wq, wsf, _) in cases[1:]:
        assert np.array_equal(wq, cases[0][1]) and np.array_equal(wsf, cases[0][2])
    work = torch.empty(iq.prepare_q_host_workspace_bytes(M), dtype=torch.uint8, device="cuda")
    outs = []
    with _chunk_rows(256):
        for x, _, _, pos in cases:
            lat, p = _host_inputs(x, pos)
            outs.append(iq.prepare_q_host(lat, w, ws, p, workspace=work))
    torch.cuda.current_stream().synchronize()
    for (x, wq, wsf, pos), (q, sf) in zip(cases, outs):
        oq, osf, oz = O.prepare_q(x, wq, wsf, pos)
        check_fp4(q.numpy(), sf.numpy(), oq, osf, oz)


def test_host_entry_errors(cuda_device):
    iq = _iq()
    L = iq.lib()
    M = 64
    x, wq, wsf, pos = W.decode_chain(M)
    w, ws = _weights(wq, wsf)
    lat, p = _host_inputs(x, pos)
    q = torch.empty((M, 4096), dtype=torch.uint8).pin_memory()
    sf = torch.empty((M, 256), dtype=torch.uint8).pin_memory()
    need = iq.prepare_q_host_workspace_bytes(M)
    work = torch.empty(need, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def call(lat_ptr=lat.data_ptr(), pos_ptr=p.data_ptr(), q_ptr=q.data_ptr(), ws_bytes=need, m=M, fmt=0):
        return L.iq_prepare_q_host(lat_ptr, m, w.data_ptr(), ws.data_ptr(), pos_ptr, fmt, q_ptr, sf.data_ptr(),
                                   work.data_ptr(), ws_bytes, stream)

    pageable = np.zeros((M, 1536), dtype=np.uint16)
    pageable_q = np.zeros((M, 4096), dtype=np.uint8)
    assert call(lat_ptr=pageable.ctypes.data) == -1          # IQ_ERR_ARG: pageable latent
    assert call(q_ptr=pageable_q.ctypes.data) == -1          # IQ_ERR_ARG: pageable output
    assert call(ws_bytes=need - 1) == -6                     # IQ_ERR_WORKSPACE
    assert call(fmt=7) == -1                                 # unknown FP4 format
    assert call(m=0) == 0                                    # nothing to do
    assert call() == 0
    torch.cuda.current_stream().synchronize()
    check_fp4(q.numpy(), sf.numpy(), *O.prepare_q(x, wq, wsf, pos))
    with pytest.raises(ValueError):
        iq.prepare_q_host(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16), w, ws, p)

