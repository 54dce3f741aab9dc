"""GPU parity of the indexer-Q preparation path (iq_prepare_q and friends)
against the CPU oracle, with the rules of tests/parity.py."""

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


def _dev(x, pos, wq, wsf):
    lat = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return (lat, torch.from_numpy(wq).cuda(), torch.from_numpy(wsf).cuda(), torch.from_numpy(pos).cuda())


def _run(x, wq, wsf, pos, debug=True):
    iq = _iq()
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    out = iq.prepare_q(lat, w, ws, p, debug=debug)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in out]


def _check_all(x, wq, wsf, pos):
    q, sf, z = _run(x, wq, wsf, pos)
    oq, osf, oz = O.prepare_q(x, wq, wsf, pos)
    worst = check_prequant(z, oz)
    stats = check_fp4(q, sf, oq, osf, oz)
    stats["prequant_worst"] = worst
    return stats


def test_tiny_chain_16_tokens(cuda_device):
    stats = _check_all(*W.tiny_chain(16))
    assert stats["equal_fraction"] >= 0.9999


@pytest.mark.parametrize("M", [1, 4, 5, 8, 16, 127, 129, 300])
def test_odd_token_counts(cuda_device, M):
    _check_all(*W.chain_workload(M, seed=100 + M, outlier_p=0.001, outlier_scale=50.0))


def test_prefill_4632_tokens_full_compare(cuda_device):
    stats = _check_all(*W.prefill_chain(4632))
    print("prefill 4632:", stats)


@pytest.mark.parametrize("M", [128, 512, 1024])
def test_sweep_points_full_compare(cuda_device, M):
    _check_all(*W.sweep_chain(M))


@pytest.mark.parametrize("M", [16384, 65536])
def test_sweep_points_sampled_rows(cuda_device, M):
    """Large sweep points: the GPU runs the whole problem; the oracle checks a
    seeded sample of rows (every M tile's first and last row among them)."""
    x, wq, wsf, pos = W.sweep_chain(M)
    q, sf, z = _run(x, wq, wsf, pos)
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([rng.choice(M, 96, replace=False), [0, 127, 128, M - 1]]))
    oq, osf, oz = O.prequant_q_rows(x, wq, wsf, pos, rows)
    check_prequant(z[rows], oz)
    check_fp4(q[rows], sf[rows], oq, osf, oz)
    # properties that hold on every row: scale bytes within the reachable range
    assert sf.min() >= 112 and sf.max() < 160


@pytest.mark.parametrize("M", [4633, 4864, 4865])
def test_prefill_tails_sampled_rows(cuda_device, M):
    """Token counts around the prefill size: one row past 4632 (a twentieth
    256-row block with one row), exactly 19 blocks, and one row past that.
    Sampled rows include every 128-row tile edge of the last two blocks."""
    x, wq, wsf, pos = W.chain_workload(M, seed=M, outlier_p=0.001, outlier_scale=50.0)
    q, sf, z = _run(x, wq, wsf, pos)
    rng = np.random.default_rng(M)
    edges = [e for b in range(4352, M + 1, 128) for e in (b - 1, b) if e < M]
    rows = np.unique(np.concatenate([rng.choice(M, 48, replace=False), edges, [0, M - 1]]))
    oq, osf, oz = O.prequant_q_rows(x, wq, wsf, pos, rows)
    check_prequant(z[rows], oz)
    check_fp4(q[rows], sf[rows], oq, osf, oz)


def test_nondebug_equals_debug_and_stage_two_alone(cuda_device):
    iq = _iq()
    x, wq, wsf, pos = W.chain_workload(777, seed=9, outlier_p=0.005, outlier_scale=100.0)
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    q1, s1 = iq.prepare_q(lat, w, ws, p)
    q2, s2, _ = iq.prepare_q(lat, w, ws, p, debug=True)
    xq, xs = iq.fp8_quant_1x128_ue8m0(lat)
    q3, s3 = iq.gemm_rope_hadamard_fp4(xq, xs, w, ws, p)
    torch.cuda.synchronize()
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
    assert torch.equal(q1, q3) and torch.equal(s1, s3)
    check_fp8(xq.cpu().numpy(), xs.cpu().numpy(), *O.fp8_quant_1x128_ue8m0(x))


def test_workspace_holds_stage_one_outputs(cuda_device):
    iq = _iq()
    M = 70
    x, wq, wsf, pos = W.tiny_chain(M)
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    nbytes = iq.prepare_q_workspace_bytes(M)
    work = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    iq.prepare_q(lat, w, ws, p, workspace=work)
    torch.cuda.synchronize()
    off = (M * 1536 + 255) // 256 * 256
    codes = work[:M * 1536].view(M, 1536).cpu().numpy()
    words = work[off:off + 3 * 72 * 4].view(torch.int32).view(3, 72).cpu().numpy()
    check_fp8(codes, words, *O.fp8_quant_1x128_ue8m0(x))


def test_zero_latent(cuda_device):
    x, wq, wsf, pos = W.tiny_chain(9)
    x = np.zeros_like(x)
    q, sf, z = _run(x, wq, wsf, pos)
    # every code decodes to zero (exact zeros may carry either sign: RoPE
    # forms 0 * cos with cos < 0), every block takes the floor scale 2^-15
    assert np.all((q & 0x77) == 0) and np.all(sf == 112) and np.all(z == 0)
    check_fp4(q, sf, *O.prepare_q(x, wq, wsf, pos))


def test_cuda_graph_replay_matches_eager(cuda_device):
    iq = _iq()
    for M in (1, 8, 32, 64, 200):
        x, wq, wsf, pos = W.decode_chain(M)
        lat, w, ws, p = _dev(x, pos, wq, wsf)
        work = torch.empty(iq.prepare_q_workspace_bytes(M), dtype=torch.uint8, device="cuda")
        q = torch.empty((M, 4096), dtype=torch.uint8, device="cuda")
        s = torch.empty((M, 256), dtype=torch.uint8, device="cuda")
        iq.prepare_q(lat, w, ws, p, q_fp4=q, q_sf=s, workspace=work)     # eager (also sets up the device)
        torch.cuda.synchronize()
        qe, se = q.clone(), s.clone()
        q.zero_()
        s.zero_()
        g = torch.cuda.CUDAGraph()
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                iq.prepare_q(lat, w, ws, p, q_fp4=q, q_sf=s, workspace=work)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert torch.equal(q, qe) and torch.equal(s, se), M
        oq, osf, oz = O.prepare_q(x, wq, wsf, pos)
        check_fp4(qe.cpu().numpy(), se.cpu().numpy(), oq, osf, oz)


def test_prepare_q_argument_errors(cuda_device):
    iq = _iq()
    L = iq.lib()
    M = 8
    x, wq, wsf, pos = W.tiny_chain(M)
    lat, w, ws, p = _dev(x, pos, wq, wsf)
    q = torch.empty((M, 4096), dtype=torch.uint8, device="cuda")
    s = torch.empty((M, 256), dtype=torch.uint8, device="cuda")
    need = L.iq_prepare_q_workspace(M)
    work = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    args = [lat.data_ptr(), M, w.data_ptr(), ws.data_ptr(), p.data_ptr(), q.data_ptr(), s.data_ptr()]
    assert L.iq_prepare_q(*args, work.data_ptr(), need - 1, st) == -6
    assert L.iq_prepare_q(*args, work.data_ptr() + 16, need, st) == -2
    bad = list(args)
    bad[0] += 2
    assert L.iq_prepare_q(*bad, work.data_ptr(), need, st) == -2
    bad = list(args)
    bad[2] = None
    assert L.iq_prepare_q(*bad, work.data_ptr(), need, st) == -1
    zero = list(args)
    zero[1] = 0
    assert L.iq_prepare_q(*zero, None, 0, st) == 0
    assert L.iq_prepare_q(*args, work.data_ptr(), need, st) == 0
    torch.cuda.synchronize()


def test_device_status_word_is_clean(cuda_device):
    """No bounded wait gave up in any launch of this session."""
    assert _iq().device_status() == 0


@pytest.mark.parametrize("M", [5, 100, 300])
def test_negative_and_large_positions(cuda_device, M):
    """The header allows any position with |p| < 2^24: negative positions and
    positions far beyond the pages' 163840 rotate like any other, on the
    small-M route (M = 5: 64 token columns, M = 100: 128) and the CTA-pair
    route (M = 300)."""
    x, wq, wsf, pos = W.chain_workload(M, seed=4000 + M, outlier_p=0.001, outlier_scale=50.0)
    rng = np.random.default_rng(M)
    pos = rng.integers(-(1 << 24) + 1, 1 << 24, size=M).astype(np.int32)
    pos[:4] = [-1, -163840, (1 << 24) - 1, -(1 << 24) + 1]
    q, sf, z = _run(x, wq, wsf, pos)
    oq, osf, oz = O.prepare_q(x, wq, wsf, pos)
    check_prequant(z, oz)
    check_fp4(q, sf, oq, osf, oz)


def test_fp4_scale_flips_over_the_configs(cuda_device):
    """Blocks whose FP4 scale byte differs from the oracle's (allowed only next
    to the scale rule's decision boundary, their codes then checked under the
    GPU's own scale) over the chain configurations: the tiny chain, the decode
    batches, the 4632-token prefill and the sweep points up to 1024 tokens.
    Such blocks must stay rare; the count is printed."""
    cases = [W.tiny_chain(16)] + [W.decode_chain(m) for m in (1, 8, 32, 64)] + [W.prefill_chain(4632)]
    cases += [W.sweep_chain(m) for m in (128, 512, 1024)]
    flips = blocks = zero_flips = codes = 0
    for x, wq, wsf, pos in cases:
        q, sf = _run(x, wq, wsf, pos, debug=False)
        oq, osf, oz = O.prepare_q(x, wq, wsf, pos)
        st = check_fp4(q, sf, oq, osf, oz)
        flips += st["scale_mismatch_blocks"]
        zero_flips += st["signed_zero_flips"]
        codes += st["code_mismatches"]
        blocks += osf.size
    print(f"FP4 scale flips {flips} of {blocks} blocks; one-step code mismatches {codes}; +0/-0 flips {zero_flips}")
    assert flips <= max(1, blocks // 100000)
