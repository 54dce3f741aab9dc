"""Writes stay inside their buffers: every output, scale array and workspace
is a view into a larger buffer whose bytes before and after it hold a canary
pattern, and the canaries must be intact after the call.  Covers the
quantizer (ragged K), both GEMM routes at ragged M (the bulk tensor stores
clip at row M; the scale stores are per row) and the host-buffer entry with a
ragged last chunk.
"""

import contextlib

import numpy as np
import pytest
import torch

from fp4_fp8_quant_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CANARY = 0xA5
PAD = 4096          # bytes of canary on each side; a multiple of 256 keeps every view aligned


def _iq():
    from fp4_fp8_quant_gb300 import iq
    return iq


class Guarded:
    """A uint8 buffer of `nbytes` with PAD canary bytes on both sides."""

    def __init__(self, nbytes, device="cuda", pinned=False):
        self.n = nbytes
        if device == "cpu":
            self.buf = torch.full((nbytes + 2 * PAD,), CANARY, dtype=torch.uint8)
            if pinned:
                self.buf = self.buf.pin_memory()
        else:
            self.buf = torch.full((nbytes + 2 * PAD,), CANARY, dtype=torch.uint8, device=device)

    def view(self, dtype=torch.uint8, shape=None):
        v = self.buf[PAD:PAD + self.n].view(dtype)
        return v if shape is None else v.view(shape)

    def intact(self):
        b = self.buf.cpu().numpy()
        return bool(np.all(b[:PAD] == CANARY) and np.all(b[PAD + self.n:] == CANARY))


@contextlib.contextmanager
def _route(threshold):
    iq = _iq()
    old = iq.set_small_m_threshold(threshold)
    try:
        yield
    finally:
        iq.set_small_m_threshold(old)


def _weights(wq, wsf):
    return torch.from_numpy(wq).cuda(), torch.from_numpy(wsf).cuda()


@pytest.mark.parametrize("M,K", [(1, 128), (5, 640), (130, 1536), (33, 7168)])
def test_quantizer_writes_stay_inside(cuda_device, M, K):
    iq = _iq()
    x = torch.randn((M, K), device="cuda").to(torch.bfloat16)
    y = Guarded(M * K)
    words = iq.scale_words(M, K)
    s = Guarded(words * 4)
    iq.fp8_quant_1x128_ue8m0(x, y=y.view(shape=(M, K)), scales=s.view(torch.int32, ((K + 511) // 512, -1)))
    torch.cuda.synchronize()
    assert y.intact() and s.intact()


@pytest.mark.parametrize("M,threshold", [(1, 128), (37, 128), (64, 128), (37, 0), (65, 64), (65, 128), (100, 128),
                                         (128, 128), (128, 0), (300, 128), (4633, 128)])
def test_prepare_q_writes_stay_inside(cuda_device, M, threshold):
    iq = _iq()
    x, wq, wsf, pos = W.decode_chain(M)
    w, ws = _weights(wq, wsf)
    lat = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    p = torch.from_numpy(pos).cuda()
    q = Guarded(M * 4096)
    sf = Guarded(M * 256)
    work = Guarded(iq.prepare_q_workspace_bytes(M))
    z = Guarded(M * 8192 * 4)
    with _route(threshold):
        iq.prepare_q(lat, w, ws, p, q_fp4=q.view(shape=(M, 4096)), q_sf=sf.view(shape=(M, 256)),
                     workspace=work.view(), q_prequant=z.view(torch.float32, (M, 8192)))
    torch.cuda.synchronize()
    assert q.intact() and sf.intact() and work.intact() and z.intact()
    assert iq.device_status() == 0


@pytest.mark.parametrize("fmt", ["mx_ocp", "nv"])
def test_fp4_variant_writes_stay_inside(cuda_device, fmt):
    iq = _iq()
    M = 77
    x, wq, wsf, pos = W.decode_chain(M)
    w, ws = _weights(wq, wsf)
    lat = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    p = torch.from_numpy(pos).cuda()
    cols = 512 if fmt == "nv" else 256
    for threshold in (0, 128):
        q = Guarded(M * 4096)
        sf = Guarded(M * cols)
        with _route(threshold):
            iq.prepare_q(lat, w, ws, p, q_fp4=q.view(shape=(M, 4096)), q_sf=sf.view(shape=(M, cols)),
                         fp4_format=fmt)
        torch.cuda.synchronize()
        assert q.intact() and sf.intact()


def test_host_entry_writes_stay_inside(cuda_device):
    iq = _iq()
    M = 300                                   # chunks of 256 rows: 256 + 44 (small-M route)
    x, wq, wsf, pos = W.decode_chain(M)
    w, ws = _weights(wq, wsf)
    lat = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    p = torch.from_numpy(pos).pin_memory()
    q = Guarded(M * 4096, device="cpu", pinned=True)
    sf = Guarded(M * 256, device="cpu", pinned=True)
    work = Guarded(iq.prepare_q_host_workspace_bytes(M))
    old = iq.set_host_chunk_rows(256)
    try:
        iq.prepare_q_host(lat, w, ws, p, q_fp4=q.view(shape=(M, 4096)), q_sf=sf.view(shape=(M, 256)),
                          workspace=work.view())
        torch.cuda.synchronize()
    finally:
        iq.set_host_chunk_rows(old)
    assert q.intact() and sf.intact() and work.intact()
    assert iq.device_status() == 0
