"""GPU parity of the downstream indexer (iq_indexer_logits, iq_indexer_topk)
against the CPU oracle, with the rules of tests/parity.py."""

import numpy as np
import pytest
import torch

from oracle import iq_oracle as O
from fp4_fp8_quant_gb300 import workloads as W
from tests.parity import check_logits, check_topk_vs_oracle_scores

pytestmark = pytest.mark.gpu

SENTINEL = 12345.0


def _iq():
    from fp4_fp8_quant_gb300 import iq
    return iq


def _dev(*arrays):
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrays]


def _run_logits(q, qs, k, ks, w, L, ld_pad=0):
    iq = _iq()
    M, N = q.shape[0], k.shape[0]
    dq, dqs, dk, dks, dw, dL = _dev(q, qs, k, ks, w, L)
    out = torch.full((M, N + ld_pad), SENTINEL, dtype=torch.float32, device="cuda")
    iq.indexer_logits(dq, dqs, dk, dks, dw, dL, logits=out[:, :N] if ld_pad else out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("M,N,causal", [(1, 1, False), (2, 5, False), (3, 128, True), (5, 200, True),
                                        (64, 300, True), (129, 1000, True), (37, 513, False), (16, 4632, True)])
def test_logits_match_oracle(cuda_device, M, N, causal):
    q, qs, k, ks, w, L = W.indexer_inputs(M, N, seed=M * 7 + N, causal=causal)
    got = _run_logits(q, qs, k, ks, w, L, ld_pad=3)
    ora = O.indexer_logits(q, qs, k, ks, w, L)
    mag = O.indexer_logit_magnitude(q, qs, k, ks, w)
    check_logits(got[:, :N], ora, mag, L)
    for t in range(M):   # entries past L[t] and the padding columns are not written
        assert np.all(got[t, L[t]:] == SENTINEL)
    assert _iq().device_status() == 0


def test_logits_lengths_edge_cases(cuda_device):
    M, N = 9, 300
    q, qs, k, ks, w, _ = W.indexer_inputs(M, N, seed=11, causal=False)
    L = np.array([0, -5, 1, 127, 128, 129, 299, 300, 10 ** 6], np.int32)
    got = _run_logits(q, qs, k, ks, w, L)
    ora = O.indexer_logits(q, qs, k, ks, w, np.clip(L, 0, N))
    mag = O.indexer_logit_magnitude(q, qs, k, ks, w)
    check_logits(got, ora, mag, np.clip(L, 0, N))
    assert np.all(got[0] == SENTINEL) and np.all(got[1] == SENTINEL)


def _topk(logits, L, k, N=None):
    iq = _iq()
    dl, dL = _dev(np.asarray(logits, np.float32), np.asarray(L, np.int32))
    out = iq.indexer_topk(dl, dL, k, N=N)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("N", [5000, 5001])
@pytest.mark.parametrize("k", [1, 7, 64, 2048])
def test_topk_selection_is_exact_on_given_scores(cuda_device, k, N):
    """The selection on arbitrary float32 scores (many ties, +-0, -inf, wide
    ranges) equals the oracle's selection on the same scores.  N = 5001 makes
    every row but the first start off a 16-byte boundary (the kernel's
    one-key-per-access path), N = 5000 keeps all rows aligned."""
    rng = np.random.default_rng(k)
    M = 12
    s = rng.integers(-20, 20, (M, N)).astype(np.float32)                   # heavy ties
    s[1] = rng.standard_normal(N).astype(np.float32) * np.float32(1e30)
    s[2] = np.where(rng.random(N) < 0.5, np.float32(0.0), np.float32(-0.0))  # only signed zeros
    s[3, ::3] = -np.inf
    s[4] = rng.standard_normal(N).astype(np.float32) * np.exp(rng.uniform(-40, 40, N)).astype(np.float32)
    s[5] = np.float32(1.0)                                                  # all equal
    L = np.array([N, N, N, N, N, N, 0, 1, k, k + 1, 4999, 2 * k], np.int32)
    got = _topk(s, L, k)
    want = O.indexer_topk(s.astype(np.float64), L, k)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("N", [20000, 50001])
def test_topk_long_rows_are_exact(cuda_device, N):
    """Rows longer than the 256-thread instance's row cache (12288 keys): up to
    49152 keys the 1024-thread instance caches them (N = 20000), beyond that
    every pass reads them again (N = 50001, rows also off 16-byte
    boundaries); with and without ties in the first digit's threshold bin."""
    rng = np.random.default_rng(77)
    M, k = 5, 2048
    s = rng.standard_normal((M, N)).astype(np.float32)
    s[1] = rng.integers(-3, 4, N).astype(np.float32)       # a few values: the threshold bin overflows the gather
    s[2] = np.float32(2.0)
    s[3, 5000:] = -np.inf
    L = np.array([N, N, N, 15000, 12289], np.int32)
    got = _topk(s, L, k)
    want = O.indexer_topk(s.astype(np.float64), L, k)
    assert np.array_equal(got, want)


def test_indexer_prefill_chain_end_to_end(cuda_device):
    """Q from iq_prepare_q on the 4632-token prefill workload, a 4632-key
    cache, causal lengths, top-2048: sampled rows of the logits against the
    oracle, the whole selection against the oracle's selection on the GPU's
    scores, and the sampled rows against the oracle's scores (boundary rule)."""
    iq = _iq()
    M = N = 4632
    kk = 2048
    x, wq, wsf, pos = W.prefill_chain(M)
    lat = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    q, qs = iq.prepare_q(lat, torch.from_numpy(wq).cuda(), torch.from_numpy(wsf).cuda(), torch.from_numpy(pos).cuda())
    k, ks = W.indexer_keys(N, seed=5)
    w = W.indexer_weights(M, seed=6)
    L = (pos + 1).astype(np.int32)
    dk, dks, dw, dL = _dev(k, ks, w, L)
    logits = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    iq.indexer_logits(q, qs, dk, dks, dw, dL, logits=logits)
    idx = iq.indexer_topk(logits, dL, kk)
    torch.cuda.synchronize()
    qh, qsh, lg, ih = q.cpu().numpy(), qs.cpu().numpy(), logits.cpu().numpy(), idx.cpu().numpy()
    visible = np.arange(N)[None, :] < L[:, None]
    assert not np.isnan(lg[visible]).any(), "some visible scores were not written"
    assert np.isnan(lg[~visible]).all(), "scores past a query's length were written"
    want = O.indexer_topk(np.where(np.arange(N)[None, :] < L[:, None], lg.astype(np.float64), -np.inf), L, kk)
    assert np.array_equal(ih, want)
    rows = np.unique(np.concatenate([np.random.default_rng(1).choice(M, 24, replace=False), [0, 2047, 2048, M - 1]]))
    ora = O.indexer_logits(qh[rows], qsh[rows], k, ks, w[rows], L[rows])
    mag = O.indexer_logit_magnitude(qh[rows], qsh[rows], k, ks, w[rows])
    check_logits(lg[rows], ora, mag, L[rows])
    differing = check_topk_vs_oracle_scores(ih[rows], ora, mag, L[rows], kk)
    print(f"top-k rows whose set differs from the float64 oracle's at the threshold: {differing} of {len(rows)}")
    assert iq.device_status() == 0


def test_indexer_argument_errors(cuda_device):
    iq = _iq()
    L_ = iq.lib()
    st = torch.cuda.current_stream().cuda_stream
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    assert L_.iq_indexer_logits(p, p, 0, p, p, 5, p, p, p, 5, st) == 0
    assert L_.iq_indexer_logits(p, p, -1, p, p, 5, p, p, p, 5, st) == -1
    assert L_.iq_indexer_logits(p, p, 2, p, p, 5, p, p, p, 4, st) == -1           # ld < N
    assert L_.iq_indexer_logits(p + 8, p, 2, p, p, 5, p, p, p, 5, st) == -2        # q_fp4 not 16-byte aligned
    assert L_.iq_indexer_topk(p, 5, 2, 5, p, 0, p, st) == -1                       # k < 1
    assert L_.iq_indexer_topk(p + 2, 5, 2, 5, p, 3, p, st) == -2
    torch.cuda.synchronize()


@pytest.mark.parametrize("causal", [True, False])
def test_logits_every_visible_entry_written_large(cuda_device, causal):
    """4632 queries x 4632 keys (the prefill size), random codes: every
    visible score is written exactly where it belongs (the output starts as
    NaN), sampled rows match the oracle, and no wait gave up."""
    M = N = 4632
    q, qs, k, ks, w, L = W.indexer_inputs(M, N, seed=21, causal=causal)
    dq, dqs, dk, dks, dw, dL = _dev(q, qs, k, ks, w, L)
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    _iq().indexer_logits(dq, dqs, dk, dks, dw, dL, logits=out)
    lg = out.cpu().numpy()
    visible = np.arange(N)[None, :] < L[:, None]
    assert not np.isnan(lg[visible]).any() and np.isnan(lg[~visible]).all()
    rows = np.unique(np.concatenate([np.random.default_rng(2).choice(M, 16, replace=False), [0, 1, M - 2, M - 1]]))
    ora = O.indexer_logits(q[rows], qs[rows], k, ks, w[rows], L[rows])
    mag = O.indexer_logit_magnitude(q[rows], qs[rows], k, ks, w[rows])
    check_logits(lg[rows], ora, mag, L[rows])
    assert _iq().device_status() == 0
