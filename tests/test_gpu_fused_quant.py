"""The quantizer fused into the CTA-pair GEMM kernel (iq_set_quant_fusion:
one launch per call on that route; off by default, switched on here).  Its FP8 codes and scale words must be the stand-alone
quantizer's bit for bit, so every output must equal the two-launch chain's
byte for byte; the progress flags that order the kernel's loads behind its
own quantizing warps must work from a workspace holding anything, keep it
reusable, and survive graph replays with new inputs; and delayed signals must
only delay the loads (TensorRT-LLM PR "Fuse DeepSeek-V4 Indexer Q projection
with CuTe DSL", sequence diagram: the quantization and the GEMM as one fused
operation)."""

import contextlib

import numpy as np
import pytest
import torch

from oracle import iq_oracle as O
from fp4_fp8_quant_gb300 import workloads as W
from tests.parity import check_fp4, check_fp8, check_prequant

pytestmark = pytest.mark.gpu


def _iq():
    from fp4_fp8_quant_gb300 import iq
    return iq


@contextlib.contextmanager
def _fusion(on):
    """Fusion on or off, with every token count on the CTA-pair route (the
    fused launch exists only there)."""
    iq = _iq()
    prev = iq.set_quant_fusion(on)
    route = iq.set_small_m_threshold(0)
    try:
        yield
    finally:
        iq.set_quant_fusion(prev)
        iq.set_small_m_threshold(route)


def _dev(x, pos, wq, wsf):
    lat = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return lat, torch.from_numpy(wq).cuda(), torch.from_numpy(wsf).cuda(), torch.from_numpy(pos).cuda()


def _regions(M, work):
    """The workspace's FP8 latent, its scale words and the flags' epoch word."""
    off = (M * 1536 + 255) // 256 * 256
    m_al = (M + 3) // 4 * 4
    coff = (off + 3 * m_al * 4 + 255) // 256 * 256
    codes = work[:M * 1536].view(M, 1536)
    words = work[off:off + 3 * m_al * 4].view(torch.int32).view(3, m_al)
    epoch = work[coff:coff + 8].view(torch.int64)
    return codes, words, epoch


def _call(iq, lat, w, ws, p, work, fmt="mx", debug=True):
    return iq.prepare_q(lat, w, ws, p, workspace=work, fp4_format=fmt, debug=debug)


@pytest.mark.parametrize("M", [65, 100, 300, 777, 2085, 4632])
def test_fused_equals_two_launches_and_oracle(cuda_device, M):
    iq = _iq()
    x, wq, wsf, pos = W.chain_workload(M, seed=900 + M, outlier_p=0.002, outlier_scale=80.0)
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    nbytes = iq.prepare_q_workspace_bytes(M)
    work_f = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    work_u = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    with _fusion(True):
        fused = _call(iq, lat, w, ws, p, work_f)
        e0 = int(_regions(M, work_f)[2].item())
        again = _call(iq, lat, w, ws, p, work_f)
    with _fusion(False):
        chain = _call(iq, lat, w, ws, p, work_u)
    torch.cuda.synchronize()
    for a, b, c in zip(fused, chain, again):
        assert torch.equal(a, b) and torch.equal(a, c)
    cf, wf, epoch = _regions(M, work_f)
    cu, wu, _ = _regions(M, work_u)
    assert torch.equal(cf, cu) and torch.equal(wf, wu)
    assert (int(epoch.item()) - e0) % (1 << 64) == 1, "each call advances the epoch once"
    check_fp8(cf.cpu().numpy(), wf.cpu().numpy(), *O.fp8_quant_1x128_ue8m0(x))
    oq, osf, oz = O.prepare_q(x, wq, wsf, pos)
    check_prequant(fused[2].cpu().numpy(), oz)
    check_fp4(fused[0].cpu().numpy(), fused[1].cpu().numpy(), oq, osf, oz)
    assert iq.device_status() == 0


@pytest.mark.parametrize("fmt", ["mx_ocp", "nv"])
def test_fused_variants_equal_two_launches(cuda_device, fmt):
    iq = _iq()
    M = 1000
    x, wq, wsf, pos = W.chain_workload(M, seed=31, outlier_p=0.002, outlier_scale=80.0)
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    with _fusion(True):
        fused = _call(iq, lat, w, ws, p, None, fmt)
    with _fusion(False):
        chain = _call(iq, lat, w, ws, p, None, fmt)
    torch.cuda.synchronize()
    for a, b in zip(fused, chain):
        assert torch.equal(a, b)
    assert iq.device_status() == 0


def test_garbage_workspace_and_reuse(cuda_device):
    """A workspace full of random bytes, then the same workspace again with
    new inputs (the previous call's flags must not count), then with a
    different token count (the flags move with M)."""
    iq = _iq()
    rng = np.random.default_rng(5)
    nbytes = iq.prepare_q_workspace_bytes(4632)
    work = torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8)).cuda()
    for M, seed in ((4632, 1), (4632, 2), (1111, 3)):
        x, wq, wsf, pos = W.chain_workload(M, seed=seed, outlier_p=0.001, outlier_scale=50.0)
        lat, w, ws, p = _dev(x, pos, wq, wsf)
        with _fusion(True):
            q, sf = iq.prepare_q(lat, w, ws, p, workspace=work)
        with _fusion(False):
            q2, sf2 = iq.prepare_q(lat, w, ws, p)
        torch.cuda.synchronize()
        assert torch.equal(q, q2) and torch.equal(sf, sf2), (M, seed)
    assert iq.device_status() == 0


def test_delayed_rows_only_delay(cuda_device):
    """Each wave's signal held back by 200 us: the loads wait for it and the
    bytes stay the same."""
    iq = _iq()
    M = 3000
    x, wq, wsf, pos = W.chain_workload(M, seed=77, outlier_p=0.001, outlier_scale=50.0)
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    ref = _call(iq, lat, w, ws, p, None)
    iq.debug_delay_quant_ns(200_000)
    try:
        with _fusion(True):
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            start.record()
            slow = _call(iq, lat, w, ws, p, None)
            end.record()
    finally:
        iq.debug_delay_quant_ns(0)
    torch.cuda.synchronize()
    assert start.elapsed_time(end) > 0.2, "the delay was applied"
    for a, b in zip(ref, slow):
        assert torch.equal(a, b)
    assert iq.device_status() == 0


def test_graph_replays_see_new_inputs(cuda_device):
    """One captured call replayed over changing latents: a stale flag from the
    previous replay would let the loads read the previous rows."""
    iq = _iq()
    M = 2000
    xs = [W.chain_workload(M, seed=40 + i, outlier_p=0.001, outlier_scale=50.0) for i in range(3)]
    _, wq, wsf, pos = xs[0]
    lat, w, ws, p = _dev(xs[0][0], pos, wq, wsf)
    work = torch.empty(iq.prepare_q_workspace_bytes(M), dtype=torch.uint8, device="cuda")
    q = torch.empty((M, 4096), dtype=torch.uint8, device="cuda")
    s = torch.empty((M, 256), dtype=torch.uint8, device="cuda")
    with _fusion(True):
        iq.prepare_q(lat, w, ws, p, q_fp4=q, q_sf=s, workspace=work)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                iq.prepare_q(lat, w, ws, p, q_fp4=q, q_sf=s, workspace=work)
    for x, _, _, _ in xs:
        new = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
        lat.copy_(new)
        g.replay()
        with _fusion(False):
            qe, se = iq.prepare_q(new, w, ws, p)
        torch.cuda.synchronize()
        assert torch.equal(q, qe) and torch.equal(s, se)
    assert iq.device_status() == 0


def test_sweep_size_sampled_rows(cuda_device):
    """16384 tokens (27 waves of tiles): sampled rows against the oracle, all
    rows against the two-launch chain."""
    iq = _iq()
    M = 16384
    x, wq, wsf, pos = W.sweep_chain(M)
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    with _fusion(True):
        q, sf = iq.prepare_q(lat, w, ws, p)
    with _fusion(False):
        q2, sf2 = iq.prepare_q(lat, w, ws, p)
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(sf, sf2)
    rows = np.unique(np.concatenate([np.random.default_rng(8).choice(M, 48, replace=False), [0, 255, 256, M - 1]]))
    oq, osf, oz = O.prequant_q_rows(x, wq, wsf, pos, rows)
    check_fp4(q.cpu().numpy()[rows], sf.cpu().numpy()[rows], oq, osf, oz)
    assert iq.device_status() == 0
