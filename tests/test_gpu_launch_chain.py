"""Back-to-back calls on one stream.  Every kernel of the path lets the next
kernel of the stream launch while it runs, and the quantizer is itself a
programmatic dependent of whatever precedes it, waiting for it before any
memory access.  Calls issued without a host synchronisation between them, on
one shared workspace, must therefore give the bytes each call gives alone,
and a quantizer whose input the immediately preceding kernel writes must read
the new values (TensorRT-LLM PR "Fuse DeepSeek-V4 Indexer Q projection with
CuTe DSL", sequence diagram: the quantization, then the GEMM on its output);
the same holds for the indexer kernels that consume the prepared Q (TokenSpeed
PR "perf(deepseek-v4): accelerate indexer Q and packed FP8 quantization",
Summary)."""

import numpy as np
import pytest
import torch

from fp4_fp8_quant_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _iq():
    from fp4_fp8_quant_gb300 import iq
    return iq


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def _inputs(M, n, seed):
    xs = [W.chain_workload(M, seed=seed + i, outlier_p=0.002, outlier_scale=60.0) for i in range(n)]
    _, wq, wsf, pos = xs[0]
    return [_bf16(x[0]) for x in xs], torch.from_numpy(wq).cuda(), torch.from_numpy(wsf).cuda(), \
        torch.from_numpy(pos).cuda()


def _alone(iq, lat, w, ws, p):
    out = iq.prepare_q(lat, w, ws, p)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("M", [1, 64, 65, 300, 4632])
def test_unsynchronised_calls_on_one_workspace(cuda_device, M):
    """Four calls in a row on the small-M or the pair route, then the same in
    a captured graph: the next call's quantizer rewrites the workspace that
    the previous call's GEMM reads."""
    iq = _iq()
    lats, w, ws, p = _inputs(M, 4, 500 + M)
    want = [_alone(iq, lat, w, ws, p) for lat in lats]
    work = torch.empty(iq.prepare_q_workspace_bytes(M), dtype=torch.uint8, device="cuda")
    outs = [(torch.empty((M, 4096), dtype=torch.uint8, device="cuda"),
             torch.empty((M, 256), dtype=torch.uint8, device="cuda")) for _ in lats]
    for lat, (q, s) in zip(lats, outs):
        iq.prepare_q(lat, w, ws, p, q_fp4=q, q_sf=s, workspace=work)
    torch.cuda.synchronize()
    for (q, s), (qw, sw) in zip(outs, want):
        assert torch.equal(q, qw) and torch.equal(s, sw)
    for q, s in outs:
        q.zero_()
        s.zero_()
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for lat, (q, s) in zip(lats, outs):
                iq.prepare_q(lat, w, ws, p, q_fp4=q, q_sf=s, workspace=work)
    g.replay()
    torch.cuda.synchronize()
    for (q, s), (qw, sw) in zip(outs, want):
        assert torch.equal(q, qw) and torch.equal(s, sw)
    assert iq.device_status() == 0


@pytest.mark.parametrize("M", [48, 2000])
def test_quantizer_sees_the_preceding_kernels_writes(cuda_device, M):
    """The latent is written by the kernel right before each call (an add
    that waits on a long reduction), with no host synchronisation."""
    iq = _iq()
    lats, w, ws, p = _inputs(M, 3, 900 + M)
    want = [_alone(iq, lat, w, ws, p) for lat in lats]
    heavy = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    lat = torch.empty_like(lats[0])
    got = []
    for x in lats:
        torch.add(x, heavy.sum().to(torch.bfloat16) * 0, out=lat)
        got.append(iq.prepare_q(lat, w, ws, p))
    torch.cuda.synchronize()
    for (q, s), (qw, sw) in zip(got, want):
        assert torch.equal(q, qw) and torch.equal(s, sw)
    assert iq.device_status() == 0


def test_stand_alone_quantizer_after_a_writer(cuda_device):
    """iq_fp8_quant_1x128_ue8m0 right after the kernel that writes its input."""
    iq = _iq()
    rng = np.random.default_rng(3)
    xs = [torch.from_numpy(rng.standard_normal((777, 7168)).astype(np.float32)).cuda().to(torch.bfloat16)
          for _ in range(3)]
    want = [iq.fp8_quant_1x128_ue8m0(x) for x in xs]
    torch.cuda.synchronize()
    heavy = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    buf = torch.empty_like(xs[0])
    got = []
    for x in xs:
        torch.add(x, heavy.sum().to(torch.bfloat16) * 0, out=buf)
        got.append(iq.fp8_quant_1x128_ue8m0(buf))
    torch.cuda.synchronize()
    for (y, s), (yw, sw) in zip(got, want):
        assert torch.equal(y, yw) and torch.equal(s, sw)


def test_prepare_then_indexer_without_synchronisation(cuda_device):
    """prepare_q -> indexer_logits -> indexer_topk, three times in a row on one
    stream with new latents and shared buffers: the logits kernel reads the
    FP4 Q and its scales that the GEMM just wrote, the top-k reads the scores
    the logits kernel just wrote (each waits for its predecessor while both
    may be resident), and every result must equal the same calls made one at
    a time with synchronisations between them."""
    iq = _iq()
    M, N = 2000, 3000
    lats, w, ws, p = _inputs(M, 3, 700)
    k_np, ks_np = W.indexer_keys(N, seed=5)
    kf, ksf = torch.from_numpy(k_np).cuda(), torch.from_numpy(ks_np).cuda()
    hw = torch.from_numpy(W.indexer_weights(M, seed=6)).cuda()
    lengths = torch.from_numpy(np.clip(np.arange(N - M, N) + 1, 0, N).astype(np.int32)).cuda()
    want = []
    for lat in lats:
        q, s = _alone(iq, lat, w, ws, p)
        lg = torch.zeros((M, N), dtype=torch.float32, device="cuda")
        iq.indexer_logits(q, s, kf, ksf, hw, lengths, logits=lg)
        torch.cuda.synchronize()
        top = iq.indexer_topk(lg, lengths, 1024)
        torch.cuda.synchronize()
        want.append((lg.clone(), top.clone()))
    q = torch.empty((M, 4096), dtype=torch.uint8, device="cuda")
    s = torch.empty((M, 256), dtype=torch.uint8, device="cuda")
    work = torch.empty(iq.prepare_q_workspace_bytes(M), dtype=torch.uint8, device="cuda")
    lg = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    got = []
    for lat in lats:
        iq.prepare_q(lat, w, ws, p, q_fp4=q, q_sf=s, workspace=work)
        iq.indexer_logits(q, s, kf, ksf, hw, lengths, logits=lg)
        top = iq.indexer_topk(lg, lengths, 1024)
        got.append((lg.clone(), top))
    torch.cuda.synchronize()
    for (lg_g, top_g), (lg_w, top_w) in zip(got, want):
        assert torch.equal(lg_g, lg_w) and torch.equal(top_g, top_w)
    assert iq.device_status() == 0


def test_mixed_routes_back_to_back(cuda_device):
    """Calls of different token counts in a row on one stream, so that each
    kernel's programmatic successor is another route or instance (both
    small-M widths and the CTA-pair kernel), eager and in a captured graph;
    every result must equal the same call made alone."""
    iq = _iq()
    Ms = [100, 64, 300, 1, 128, 4632, 65]
    cases = [_inputs(M, 1, 1300 + M) for M in Ms]
    want = [_alone(iq, lats[0], w, ws, p) for (lats, w, ws, p) in cases]
    outs = [(torch.empty((M, 4096), dtype=torch.uint8, device="cuda"),
             torch.empty((M, 256), dtype=torch.uint8, device="cuda")) for M in Ms]
    works = [torch.empty(iq.prepare_q_workspace_bytes(M), dtype=torch.uint8, device="cuda") for M in Ms]

    def issue():
        for (lats, w, ws, p), (q, s), work in zip(cases, outs, works):
            iq.prepare_q(lats[0], w, ws, p, q_fp4=q, q_sf=s, workspace=work)

    issue()
    torch.cuda.synchronize()
    for (q, s), (qw, sw) in zip(outs, want):
        assert torch.equal(q, qw) and torch.equal(s, sw)
    for q, s in outs:
        q.zero_()
        s.zero_()
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            issue()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for (q, s), (qw, sw) in zip(outs, want):
        assert torch.equal(q, qw) and torch.equal(s, sw)
    assert iq.device_status() == 0
