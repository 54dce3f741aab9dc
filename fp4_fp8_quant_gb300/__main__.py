"""Runs one case of the indexer-Q path on seeded synthetic inputs and prints
its CUDA-event time per call -- a quick check of a build, and the command the
profiles are taken with.

    python -m fp4_fp8_quant_gb300 prepare --tokens 4632 [--repeat 3] [--route auto|small|pair]
    python -m fp4_fp8_quant_gb300 quant --rows 4632 --cols 7168 [--repeat 3]
    python -m fp4_fp8_quant_gb300 indexer --queries 4632 --keys 4632 [--topk 2048] [--full] [--repeat 3]

`prepare` calls iq_prepare_q on the prefill workload when --tokens is 4632
(positions 0..M-1) and on the decode workload otherwise (random positions);
`quant` calls the FP8 1x128 quantizer on the blocks workload; `indexer` scores
random FP4 queries against a random FP4 key cache (causal unless --full) and
selects the top-k keys per query.  L2 is flushed before every call.
"""

from __future__ import annotations

import argparse
import sys

import numpy as np
import torch

from . import iq
from . import workloads as W


def _bf16(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def _time_calls(fn, repeat: int, dev) -> list[float]:
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = []
    for _ in range(repeat):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b) * 1e3)
    return out


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(prog="python -m fp4_fp8_quant_gb300")
    sub = ap.add_subparsers(dest="cmd", required=True)
    p = sub.add_parser("prepare")
    p.add_argument("--tokens", type=int, default=4632)
    p.add_argument("--repeat", type=int, default=3)
    p.add_argument("--route", choices=["auto", "small", "pair"], default="auto")
    q = sub.add_parser("quant")
    q.add_argument("--rows", type=int, default=4632)
    q.add_argument("--cols", type=int, default=7168)
    q.add_argument("--repeat", type=int, default=3)
    ix = sub.add_parser("indexer")
    ix.add_argument("--queries", type=int, default=4632)
    ix.add_argument("--keys", type=int, default=4632)
    ix.add_argument("--topk", type=int, default=2048)
    ix.add_argument("--full", action="store_true")
    ix.add_argument("--repeat", type=int, default=3)
    args = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)

    if args.cmd == "prepare":
        M = args.tokens
        x, wq, wsf, pos = W.prefill_chain(M) if M == 4632 else W.decode_chain(M)
        lat = _bf16(x, dev)
        w, ws, p_ = torch.from_numpy(wq).to(dev), torch.from_numpy(wsf).to(dev), torch.from_numpy(pos).to(dev)
        q4 = torch.empty((M, iq.Q_DIM // 2), dtype=torch.uint8, device=dev)
        sf = torch.empty((M, iq.Q_DIM // 32), dtype=torch.uint8, device=dev)
        work = torch.empty(max(1, iq.prepare_q_workspace_bytes(M)), dtype=torch.uint8, device=dev)
        threshold = {"auto": None, "small": iq.SMALL_M_MAX, "pair": 0}[args.route]
        old = iq.set_small_m_threshold(threshold) if threshold is not None else None
        try:
            us = _time_calls(lambda: iq.prepare_q(lat, w, ws, p_, q_fp4=q4, q_sf=sf, workspace=work),
                             args.repeat, dev)
        finally:
            if old is not None:
                iq.set_small_m_threshold(old)
        print(f"prepare M={M} route={args.route}: " + " ".join(f"{u:.2f}" for u in us) + " us per call")
    elif args.cmd == "indexer":
        M, N = args.queries, args.keys
        arrays = W.indexer_inputs(M, N, seed=1, causal=not args.full)
        q4, qs, k4, ks, w, L = (torch.from_numpy(a).to(dev) for a in arrays)
        logits = torch.empty((M, N), dtype=torch.float32, device=dev)
        idx = torch.empty((M, args.topk), dtype=torch.int32, device=dev)
        us_l = _time_calls(lambda: iq.indexer_logits(q4, qs, k4, ks, w, L, logits=logits), args.repeat, dev)
        us_t = _time_calls(lambda: iq.indexer_topk(logits, L, args.topk, indices=idx), args.repeat, dev)
        print(f"indexer {M}x{N} {'full' if args.full else 'causal'}: logits " + " ".join(f"{u:.2f}" for u in us_l)
              + f" us; top-{args.topk} " + " ".join(f"{u:.2f}" for u in us_t) + " us per call")
    else:
        xb = W.quant_blocks_input(args.rows, args.cols, seed=1)
        X = _bf16(xb, dev)
        Y = torch.empty((args.rows, args.cols), dtype=torch.uint8, device=dev)
        S = torch.empty((-(-args.cols // 512), (args.rows + 3) // 4 * 4), dtype=torch.int32, device=dev)
        us = _time_calls(lambda: iq.fp8_quant_1x128_ue8m0(X, y=Y, scales=S), args.repeat, dev)
        print(f"quant {args.rows}x{args.cols}: " + " ".join(f"{u:.2f}" for u in us) + " us per call")
    return 0 if iq.device_status() == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
