"""Benchmark of the indexer-Q preparation path on GB300.

One step = one pass of the whole hot path over one batch: one iq_prepare_q
call on the BF16 latent [4632, 1536] -- the FP8 1x128 quantizer, then the
fused block-scaled FP8 GEMM with the RoPE -> Hadamard -> FP4 epilogue
(launched as the quantizer's programmatic dependent), producing packed FP4 Q
[4632, 4096] and its UE8M0 scales [4632, 256].  Inputs are seeded
synthetic data resident in HBM before the timed region; L2 is flushed (256 MB
written, then 256 MB read, so no dirty lines are left for the timed kernels to
write back) between timed steps, outside the CUDA-event intervals.  `value` is
the token count over the median of the K event-timed steps (mean, minimum and
maximum are reported beside it); the clock sampler starts first, the GPU
idles for a second, and the warm-up runs max(3, W) steps (longer warm-ups
leave GB300 in its power-capped state for the first timed steps).  The steady
state of steps run back to back over
rotating buffer sets (total over twice the L2 size; each step then also
writes back the outputs of earlier steps) is reported as `back_to_back`.  Also measured in the same run: the quantizer alone on
BF16 [4632, 7168] (GB/s against HBM), the GEMM's own launch time (for the
roofline), the end-to-end call iq_prepare_q_host on page-locked host
buffers (the latent read from and the FP4 output written to host memory
inside the timed region), steps replayed from a CUDA graph (1, 8, 32, 64, 96, 128
tokens), a token sweep (128 ... 65536), the step with each FP4 output
variant, and the CPU oracle on a bounded sample of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs an independent replica on its own GPU (the
path has no exchange step); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M_PREFILL = 4632
K_LATENT = 1536
N_Q = 8192
K_QUANT = 7168
FLOPS_PER_TOKEN = 2 * N_Q * K_LATENT
METRIC = "indexer-Q tokens/s at M=4632; FP8 quantizer GB/s vs HBM peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0            # nominal dense ratio (4.5 / 2.25 PFLOP/s)
ORACLE_SAMPLE_ROWS = 4632      # rows of the prefill workload per oracle timing (all of it)
SETTLE_S = 1.0                 # idle time between the clock sampler's first sample and the warm-up
NOMINAL_HBM_GBS = 7900.0       # HBM3e nominal bandwidth of GB300
NOMINAL_FP8_TFLOPS = 4500.0    # dense FP8 tensor nominal of GB300


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's `value` (the slowest rank's step time);
    needs the default process group when world > 1."""
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, ms_per_step: float) -> float:
    """Units all ranks processed per second, timed by the slowest rank."""
    return world * units_per_rank / (ms_per_step * 1e-3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                p = json.load(f)
            hbm = p.get("hbm_gbs")
            bf16 = p.get("bf16_tflops")
            if hbm and bf16:
                return float(hbm), float(bf16), "measured"
        except (OSError, ValueError):
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def sources_sha(paths) -> str:
    """First 16 hex digits of the SHA-256 of the listed files, concatenated in
    order (a kernel's .cu file and every header it is compiled from)."""
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_traffic(kernel_key: str):
    """DRAM bytes per launch of a kernel from the committed ncu summary, or None
    when any file the kernel is compiled from changed since the counters were
    taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f).get(kernel_key)
    if not t:
        return None
    if not all(os.path.exists(os.path.join(ROOT, rel)) for rel in t["sources"]):
        return None
    if sources_sha(t["sources"]) != t["sources_sha"]:
        return None
    return t["dram_bytes_per_launch"]


class ClockSampler:
    """nvidia-smi clocks sampled every 20 ms from the start of the chain's
    warm-up to the end of the end-to-end measurement."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return self
        # nvidia-smi takes up to a second to start (driver queries); wait for
        # its first sample so that the start-up falls outside the timed region.
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 5.0 and self.proc.poll() is None:
            if os.path.getsize(self.file.name) > 0:
                break
            time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def clocks_max_mhz(gpu_index: int) -> float:
    """The GPU's maximum SM clock (nvidia-smi), else the GB300 figure 2070."""
    try:
        out = subprocess.run(["nvidia-smi", f"--id={gpu_index}", "--query-gpu=clocks.max.sm",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10).stdout
        return float(out.strip().splitlines()[0])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError):
        return 2070.0


def cublas_fp8_tflops(dev, n: int = 8192, reps: int = 20):
    """Dense FP8 (E4M3 x E4M3 -> BF16, per-tensor scales) throughput of the
    vendor library on an n^3 GEMM, best of `reps` launches: a measured FP8
    tensor-core rate on this GPU to set beside the BF16-derived peak.  None
    when the library call is not available."""
    import torch
    try:
        a = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn)
        one = torch.ones((), device=dev, dtype=torch.float32)
        for _ in range(3):
            torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except (RuntimeError, AttributeError, TypeError):
        return None


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_sample_seconds(rows: int) -> float:
    """Times the CPU oracle (single thread) on the first `rows` tokens of the
    prefill workload in a child process, so the BLAS thread count is pinned."""
    code = (
        "import os,sys,time; sys.path.insert(0, %r)\n"
        "from fp4_fp8_quant_gb300 import workloads as W\n"
        "from oracle import iq_oracle as O\n"
        "x, wq, wsf, pos = W.prefill_chain(%d)\n"
        "x, pos = x[:%d], pos[:%d]\n"
        "t = time.perf_counter(); O.prepare_q(x, wq, wsf, pos); print(time.perf_counter() - t)\n"
    ) % (ROOT, M_PREFILL, rows, rows)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, check=True)
    return float(out.stdout.strip().splitlines()[-1])


def run_reference(args):
    """The oracle as it stands, on one host core, each step a 256-token sample
    of the prefill workload."""
    rank, world, _ = dist_info()
    if rank != 0:
        return
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    from fp4_fp8_quant_gb300 import workloads as W
    from oracle import iq_oracle as O
    rows = 256
    x, wq, wsf, pos = W.prefill_chain(M_PREFILL)
    for _ in range(args.warmup):
        O.prepare_q(x[:rows], wq, wsf, pos[:rows])
    times = []
    for i in range(args.steps):
        lo = (i * rows) % (M_PREFILL - rows)
        t = time.perf_counter()
        O.prepare_q(x[lo:lo + rows], wq, wsf, pos[lo:lo + rows])
        times.append(time.perf_counter() - t)
    per_step = sum(times) / len(times)
    value = rows / per_step
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "indexer-Q prefill chain, 4632 tokens x latent 1536 -> 64 heads x 128, "
                               "positions 0..4631 (oracle: a 256-token slice per step)", "M": M_PREFILL},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": "a 256-token slice of the 4632-token prefill workload per step, FP64 numpy, "
                                   "one thread", "cpu_model": host_cpu_model(), "host_cores": os.cpu_count()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import numpy as np
    import torch

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    from fp4_fp8_quant_gb300 import build as B
    B.build()
    from fp4_fp8_quant_gb300 import iq, workloads as W

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_src = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def flush_l2():
        # Write 256 MB, then read another 256 MB: the next step finds none of
        # its data in L2 and no dirty lines of the flush left to write back.
        flush_buf.fill_(rank & 0xFF)
        flush_src.sum()

    # Rotating buffer sets.  A timed run cycles through sets of inputs,
    # outputs and workspace whose total exceeds twice the L2 size, so every
    # step reads data that is not in L2 (each set was last touched several
    # steps before) while the steps run back to back, as repeated calls do.
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size

    def sets_for(bytes_per_set):
        return max(2, -(-2 * l2_bytes // bytes_per_set) + 1)

    def time_back_to_back(fns, steps, warmup):
        """Runs fns[i % len(fns)] for i < warmup untimed, then `steps` times
        back to back with an event between consecutive steps; returns the
        per-step intervals (ms) and the total (ms)."""
        n = len(fns)
        for i in range(warmup):
            fns[i % n]()
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        evs[0].record(stream)
        for i in range(steps):
            fns[i % n]()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
        return per, evs[0].elapsed_time(evs[-1])

    # ---------------------------------------------------- the prefill chain
    x, wq, wsf, pos = W.prefill_chain(M_PREFILL)
    M = M_PREFILL
    lat0 = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
    w0 = torch.from_numpy(wq).to(dev)
    ws = torch.from_numpy(wsf).to(dev)
    p0 = torch.from_numpy(pos).to(dev)
    ws_bytes = iq.prepare_q_workspace_bytes(M)
    set_bytes = lat0.numel() * 2 + w0.numel() + p0.numel() * 4 + M * (N_Q // 2 + N_Q // 32) + ws_bytes
    n_sets = sets_for(set_bytes)
    chain_sets = []
    for i in range(n_sets):
        chain_sets.append({"lat": lat0.clone(), "w": w0.clone(), "p": p0.clone(),
                           "q": torch.empty((M, N_Q // 2), dtype=torch.uint8, device=dev),
                           "s": torch.empty((M, N_Q // 32), dtype=torch.uint8, device=dev),
                           "work": torch.empty(ws_bytes, dtype=torch.uint8, device=dev),
                           "xq": torch.empty((M, K_LATENT), dtype=torch.uint8, device=dev),
                           "xs": torch.empty((3, (M + 3) // 4 * 4), dtype=torch.int32, device=dev)})

    def step_fn(c, fmt="mx", q=None, s=None):
        # iq_prepare_q: the quantizer, then the fused GEMM as its programmatic
        # dependent (no host or event work between the two launches).
        return lambda: iq.prepare_q(c["lat"], c["w"], ws, c["p"], q_fp4=c["q"] if q is None else q,
                                    q_sf=c["s"] if s is None else s, workspace=c["work"], fp4_format=fmt)

    steps = [step_fn(c) for c in chain_sets]
    # The clock sampler starts before the warm-up and the GPU then idles for
    # SETTLE_S, so that the sampler's start-up falls outside the timed steps
    # and the timed steps start from the state the sweep's points start from.
    # The warm-up is max(3, W) steps: on GB300 a longer one (0.1 s or more of
    # back-to-back steps) leaves the GPU in its power-capped state for the
    # next few hundred ms, where a flushed step takes ~10 % longer; sustained
    # load is what `back_to_back` reports.
    clocks = ClockSampler(local).__enter__()
    time.sleep(SETTLE_S)
    n_warm = 0
    while n_warm < max(3, args.warmup):
        steps[n_warm % n_sets]()
        n_warm += 1
    # Timed steps: each after an L2 flush (256 MB written, then 256 MB read,
    # so that no dirty lines of earlier work are left for the step to write
    # back), outside the event interval; the GPU is idle when the step is
    # launched, so the launch latency of both kernels is inside it.
    barrier()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush_l2()
        ev[i][0].record(stream)
        steps[i % n_sets]()
        ev[i][1].record(stream)
    barrier()
    t_wall = time.perf_counter() - t_wall
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_per_step = max_over_ranks(statistics.median(step_ms), world, dev)
    value = whole_job_rate(M, world, ms_per_step)
    step_stats = {"median_ms": statistics.median(step_ms), "mean_ms": sum(step_ms) / len(step_ms),
                  "min_ms": min(step_ms), "max_ms": max(step_ms), "warmup_steps_run": n_warm}

    # Steady state: the same steps back to back over the rotating sets.  Each
    # step then also writes back the dirty outputs of the steps before it
    # (the flush above moves that outside the timed interval).
    bb_ms, bb_total = time_back_to_back(steps, args.steps, n_sets)
    back_to_back = {"median_ms": statistics.median(bb_ms), "mean_ms": bb_total / len(bb_ms),
                    "tokens_per_s": M / (bb_total / len(bb_ms) * 1e-3), "buffer_sets": n_sets,
                    "bytes_per_set": set_bytes,
                    "how": f"steps back to back over {n_sets} rotating buffer sets (more than twice L2)"}

    # The fused GEMM's own launch duration (for the roofline): per timed
    # launch an L2 flush, then the quantizer (outside the interval), then the
    # GEMM between events (W from HBM, the FP8 latent in L2, as in a step).
    def flushed_ms(pre, fn, n):
        out = []
        for i in range(n):
            flush_l2()
            if pre is not None:
                pre(i)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn(i)
            b.record(stream)
            out.append((a, b))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in out]

    def k1_of(i):
        c = chain_sets[i % n_sets]
        iq.fp8_quant_1x128_ue8m0(c["lat"], y=c["xq"], scales=c["xs"])

    def k2_of(i):
        c = chain_sets[i % n_sets]
        iq.gemm_rope_hadamard_fp4(c["xq"], c["xs"], c["w"], ws, c["p"], q_fp4=c["q"], q_sf=c["s"])

    # Out of the power-capped state the back-to-back steps leave, then the
    # same short warm-up as the headline (clocks back up after the idle).
    time.sleep(SETTLE_S)
    for i in range(max(3, args.warmup)):
        k1_of(i)
        k2_of(i)
    k2_ms = flushed_ms(k1_of, k2_of, args.steps)
    k2_avg_ms = sum(k2_ms) / len(k2_ms)
    k1_ms = flushed_ms(None, k1_of, args.steps)
    k1_avg_ms = sum(k1_ms) / len(k1_ms)
    k2_bb, k2_bb_total = time_back_to_back([lambda i=i: k2_of(i) for i in range(n_sets)], args.steps, 2 * n_sets)

    hbm_peak, bf16_peak, peak_kind = load_peaks()
    fp8_peak_tflops = bf16_peak * FP8_OVER_BF16
    achieved_tflops = M * FLOPS_PER_TOKEN / (k2_avg_ms * 1e-3) / 1e12
    cublas_fp8 = cublas_fp8_tflops(dev)
    roofline = {"kernel": "gemm_rope_hadamard_fp4_kernel", "bound": "tensor", "achieved": achieved_tflops,
                "peak": fp8_peak_tflops, "unit": "TFLOP/s", "frac": achieved_tflops / fp8_peak_tflops,
                "traffic": kernel_traffic("gemm_rope_hadamard_fp4_kernel"),
                "peak_source": f"{peak_kind} bf16 x {FP8_OVER_BF16:g} (FP8/BF16 nominal ratio)",
                "avg_launch_ms": k2_avg_ms, "median_launch_ms": statistics.median(k2_ms),
                "launches": "each after an L2 flush and the quantizer, events around the GEMM alone",
                "back_to_back_avg_launch_ms": k2_bb_total / len(k2_bb),
                "flops_per_launch": M * FLOPS_PER_TOKEN,
                "frac_of_nominal_fp8": achieved_tflops / NOMINAL_FP8_TFLOPS,
                "cublas_fp8_tflops_same_run": cublas_fp8,
                "frac_of_cublas_fp8": achieved_tflops / cublas_fp8 if cublas_fp8 else None}

    # ------------------------------------- FP4 output variants (prefill step)
    # The same step with each FP4 output variant of iq_prepare_q_ex (L2
    # flushed before each timed step).
    fp4_formats = {}
    for fmt in ("mx", "mx_ocp", "nv"):
        fns = []
        for c in chain_sets:
            s_f = c["s"] if fmt != "nv" else torch.empty((M, iq.fp4_scale_bytes(fmt)), dtype=torch.uint8, device=dev)
            fns.append(step_fn(c, fmt, s=s_f))
        for f in fns:
            f()
        f_ms = flushed_ms(None, lambda i: fns[i % len(fns)](), 50)
        fp4_formats[fmt] = {"us_per_step": statistics.median(f_ms) * 1e3, "mean_us_per_step": sum(f_ms) / 50 * 1e3,
                            "tokens_per_s": M / (statistics.median(f_ms) * 1e-3),
                            "scale_bytes_per_token": iq.fp4_scale_bytes(fmt)}
        del fns

    # ------------------------------------------------- the quantizer alone
    xb = W.quant_blocks_input(M_PREFILL, K_QUANT, seed=1)
    X0 = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(dev)
    q_sets = []
    q_set_bytes = M_PREFILL * K_QUANT * 3
    for i in range(sets_for(q_set_bytes)):
        q_sets.append((X0.clone(), torch.empty((M_PREFILL, K_QUANT), dtype=torch.uint8, device=dev),
                       torch.empty(((K_QUANT + 511) // 512, (M_PREFILL + 3) // 4 * 4), dtype=torch.int32,
                                   device=dev)))
    q_fns = [(lambda t=t: iq.fp8_quant_1x128_ue8m0(t[0], y=t[1], scales=t[2])) for t in q_sets]
    for f in q_fns:
        f()
    qm = flushed_ms(None, lambda i: q_fns[i % len(q_fns)](), args.steps)
    q_ms = sum(qm) / len(qm)
    qbb, qbb_total = time_back_to_back(q_fns, args.steps, 2 * len(q_sets))
    q_bytes = M_PREFILL * K_QUANT * 3 + q_sets[0][2].numel() * 4
    q_gbs = q_bytes / (q_ms * 1e-3) / 1e9
    q_bb_gbs = q_bytes / (qbb_total / len(qbb) * 1e-3) / 1e9
    quantizer = {"workload": "BF16 [4632, 7168] -> E4M3 + packed UE8M0 scales", "value": q_gbs, "unit": "GB/s",
                 "avg_launch_ms": q_ms, "median_launch_ms": statistics.median(qm),
                 "launches": "each after an L2 flush, events around the launch",
                 "back_to_back_gbs": q_bb_gbs,
                 "back_to_back_how": f"launches back to back over {len(q_sets)} buffer sets: each also writes back "
                                     f"the previous launch's output",
                 "roofline": {"kernel": "quant_1x128_kernel", "bound": "hbm", "achieved": q_gbs, "peak": hbm_peak,
                              "unit": "GB/s", "frac": q_gbs / hbm_peak, "traffic": kernel_traffic("quant_1x128_kernel"),
                              "peak_source": peak_kind, "bytes_per_launch": q_bytes,
                              "frac_of_nominal_hbm": q_gbs / NOMINAL_HBM_GBS,
                              "back_to_back_frac": q_bb_gbs / hbm_peak}}
    del q_sets, q_fns, X0
    # ------------------------------------------- decode under graph replay
    # Decode steps (N(0,1) latent, random positions) captured in a CUDA graph
    # per token count and per route (the small-M swapped-operand kernel, the
    # default for M <= 128, and the CTA-pair kernel).  Per call: a graph of 24
    # calls replayed ~1000 calls' worth, once with the same W every call (hot
    # in L2, as a decode loop sees it) and once with W rotated over 24 copies
    # (302 MB, more than twice L2), so that every call reads W from HBM.  Also
    # the replay of a graph holding one call (includes the graph launch).
    n_rot = 24
    w_rot = [w0.clone() for _ in range(n_rot)]

    def graph_us_per_call(calls, total):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        for c in calls:
            c()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for c in calls:
                    c()
        reps = max(1, total // len(calls))
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        del g
        return a.elapsed_time(b) * 1e3 / (reps * len(calls))

    decode = {"default_route_max_tokens": iq.small_m_threshold()}
    for Md in (1, 8, 32, 64, 96, 128):
        xd, _, _, pd = W.decode_chain(Md)
        lat_d = torch.from_numpy(xd.view(np.int16)).view(torch.bfloat16).to(dev)
        pos_d = torch.from_numpy(pd).to(dev)
        q_d = torch.empty((Md, N_Q // 2), dtype=torch.uint8, device=dev)
        s_d = torch.empty((Md, N_Q // 32), dtype=torch.uint8, device=dev)
        work_d = torch.empty(iq.prepare_q_workspace_bytes(Md), dtype=torch.uint8, device=dev)

        def call(wt):
            return lambda: iq.prepare_q(lat_d, wt, ws, pos_d, q_fp4=q_d, q_sf=s_d, workspace=work_d)

        entry = {}
        for route, threshold in (("small_m", iq.SMALL_M_MAX), ("cta_pair", 0)):
            old = iq.set_small_m_threshold(threshold)
            try:
                hot = graph_us_per_call([call(w0)] * n_rot, 1000)
                cold = graph_us_per_call([call(wt) for wt in w_rot], 1000)
                one = graph_us_per_call([call(w0)], 1000)
            finally:
                iq.set_small_m_threshold(old)
            entry[route] = {"us_per_call_w_in_l2": hot, "us_per_call_w_from_hbm": cold,
                            "us_per_replay_of_one_call_graph": one,
                            "w_read_gbs_from_hbm": 12.58e6 / (cold * 1e-6) / 1e9,
                            "w_read_frac_of_hbm": 12.58e6 / (cold * 1e-6) / 1e9 / hbm_peak}
        default = "small_m" if Md <= decode["default_route_max_tokens"] else "cta_pair"
        entry["tokens_per_s"] = Md / (entry[default]["us_per_call_w_in_l2"] * 1e-6)
        decode[str(Md)] = entry
    del w_rot

    # ------------------------------------------------------ token sweep
    # Chain and quantizer-alone at each sweep point: each timed call after an
    # L2 flush, and (extra keys) back to back over rotating buffer sets whose
    # total is over twice L2; inputs generated on the device: N(0,1), 0.5% x100
    # outliers, random positions.  W is rotated with the sets.
    sweep = {}
    gen = torch.Generator(device=dev)
    gen.manual_seed(4)

    def bf16_input(rows, cols):
        t = torch.randn((rows, cols), generator=gen, device=dev)
        hit = torch.rand((rows, cols), generator=gen, device=dev) < 0.005
        return torch.where(hit, t * 100.0, t).to(torch.bfloat16)

    for Ms in (128, 512, 1024, 4632, 16384, 65536):
        lat_s = bf16_input(Ms, K_LATENT)
        pos_s = torch.randint(0, 163840, (Ms,), generator=gen, device=dev, dtype=torch.int32)
        per_set = Ms * (2 * K_LATENT + 4 + N_Q // 2 + N_Q // 32) + iq.prepare_q_workspace_bytes(Ms) + w0.numel()
        sets = []
        for i in range(sets_for(per_set)):
            sets.append({"lat": lat_s.clone(), "w": w0.clone(), "p": pos_s.clone(),
                         "q": torch.empty((Ms, N_Q // 2), dtype=torch.uint8, device=dev),
                         "s": torch.empty((Ms, N_Q // 32), dtype=torch.uint8, device=dev),
                         "work": torch.empty(iq.prepare_q_workspace_bytes(Ms), dtype=torch.uint8, device=dev)})
        fns = [step_fn(c) for c in sets]
        reps = 20 if Ms >= 16384 else 50
        for f in fns:
            f()
        c_ms = flushed_ms(None, lambda i: fns[i % len(fns)](), reps)
        cbb, cbb_total = time_back_to_back(fns, reps, 2 * len(sets))
        graph = {}
        if Ms <= 4632:
            # Per call inside a 16-call CUDA graph (no per-call launch or event
            # overhead): over the rotating sets (W and inputs from HBM), and
            # one set repeated (W in L2, as consecutive calls of a layer see it).
            graph = {"graph_us_per_call_rotated": graph_us_per_call([fns[i % len(fns)] for i in range(16)], 800),
                     "graph_us_per_call_w_in_l2": graph_us_per_call([fns[0]] * 16, 800)}
            graph["graph_frac_of_fp8_peak_rotated"] = (
                Ms * FLOPS_PER_TOKEN / (graph["graph_us_per_call_rotated"] * 1e-6) / 1e12 / fp8_peak_tflops)
        del sets, fns, lat_s
        xq_in = bf16_input(Ms, K_QUANT)
        qsets = []
        for i in range(sets_for(Ms * K_QUANT * 3)):
            qsets.append((xq_in.clone() if i else xq_in, torch.empty((Ms, K_QUANT), dtype=torch.uint8, device=dev),
                          torch.empty(((K_QUANT + 511) // 512, (Ms + 3) // 4 * 4), dtype=torch.int32, device=dev)))
        qfns = [(lambda t=t: iq.fp8_quant_1x128_ue8m0(t[0], y=t[1], scales=t[2])) for t in qsets]
        for f in qfns:
            f()
        qm = flushed_ms(None, lambda i: qfns[i % len(qfns)](), reps)
        qs_ms = sum(qm) / reps
        qbb, qbb_total = time_back_to_back(qfns, reps, 2 * len(qsets))
        qbytes = Ms * K_QUANT * 3 + qsets[0][2].numel() * 4
        del qsets, qfns, xq_in
        flops = Ms * FLOPS_PER_TOKEN
        cm = statistics.median(c_ms)
        sweep[str(Ms)] = {
            "chain_us": cm * 1e3, "chain_mean_us": sum(c_ms) / reps * 1e3, "tokens_per_s": Ms / (cm * 1e-3),
            "chain_back_to_back_us": cbb_total / reps * 1e3,
            "quant7168_back_to_back_gbs": qbytes / (qbb_total / reps * 1e-3) / 1e9,
            "chain_tflops": flops / (cm * 1e-3) / 1e12, "chain_frac_of_fp8_peak": flops / (cm * 1e-3) / 1e12 / fp8_peak_tflops,
            "quant7168_us": qs_ms * 1e3, "quant7168_gbs": qbytes / (qs_ms * 1e-3) / 1e9,
            "quant7168_frac_of_hbm": qbytes / (qs_ms * 1e-3) / 1e9 / hbm_peak, **graph}
    # The quantizer's fraction also against the best rate any of its launches
    # reached in this run (the copy-measured peak is not a ceiling for it).
    best_q = max([q_gbs] + [v["quant7168_gbs"] for v in sweep.values()])
    quantizer["roofline"]["best_kernel_gbs_in_run"] = best_q
    quantizer["roofline"]["frac_of_best_in_run"] = q_gbs / best_q
    # ------------------------------------------- downstream indexer consumer
    # The prefill step's FP4 Q (4632 tokens) scored against a 4632-key cache
    # with causal visibility (query t sees keys s <= t), then the top-2048
    # keys per query.  Each timed launch after an L2 flush.  The logits
    # kernel is bound by its per-(query, key, head) epilogue arithmetic (a
    # ReLU and a weighted add: 1.5 FP32 lane operations with packed FMAs);
    # the top-k kernel by reading the scores.
    indexer = {}
    k_np, ks_np = W.indexer_keys(M, seed=5)
    w_np = W.indexer_weights(M, seed=6)
    kdev, ksdev, wdev = (torch.from_numpy(a).to(dev) for a in (k_np, ks_np, w_np))
    len_dev = (torch.from_numpy(pos).to(dev) + 1).to(torch.int32)
    q_idx, s_idx = chain_sets[0]["q"], chain_sets[0]["s"]
    iq.prepare_q(chain_sets[0]["lat"], w0, ws, chain_sets[0]["p"], q_fp4=q_idx, q_sf=s_idx,
                 workspace=chain_sets[0]["work"])
    logits_buf = torch.empty((M, M), dtype=torch.float32, device=dev)
    topk_buf = torch.empty((M, 2048), dtype=torch.int32, device=dev)
    run_l = lambda i: iq.indexer_logits(q_idx, s_idx, kdev, ksdev, wdev, len_dev, logits=logits_buf)
    run_t = lambda i: iq.indexer_topk(logits_buf, len_dev, 2048, indices=topk_buf)
    for _ in range(3):
        run_l(0)
        run_t(0)
    il_ms = flushed_ms(None, run_l, 30)
    it_ms = flushed_ms(None, run_t, 30)
    ib_ms = flushed_ms(None, lambda i: (run_l(i), run_t(i)), 30)
    visible = int(len_dev.clamp(max=M).sum().item())
    pair_heads = visible * 64
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    alu_lane_ops_per_s = sm_count * 128 * (clocks_max_mhz(local) * 1e6)
    alu_peak_pair_heads = alu_lane_ops_per_s / 1.5
    l_avg = sum(il_ms) / len(il_ms)
    t_avg = sum(it_ms) / len(it_ms)
    topk_bytes = visible * 4 + M * 2048 * 4
    indexer = {
        "workload": "4632 queries (the prefill step's FP4 Q) x 4632 cached FP4 keys, causal, top-2048",
        "visible_pairs": visible,
        "logits_us": l_avg * 1e3, "topk_us": t_avg * 1e3, "both_us": sum(ib_ms) / len(ib_ms) * 1e3,
        "logits_roofline": {"kernel": "indexer_logits_kernel", "bound": "alu",
                            "achieved": pair_heads / (l_avg * 1e-3) / 1e12, "unit": "T pair-heads/s",
                            "peak": alu_peak_pair_heads / 1e12,
                            "frac": pair_heads / (l_avg * 1e-3) / alu_peak_pair_heads,
                            "peak_source": f"{sm_count} SMs x 128 FP32 lanes x max SM clock, 1.5 lane ops per "
                                           f"(query, key, head)",
                            "fp4_tflops": visible * 64 * 128 * 2 / (l_avg * 1e-3) / 1e12,
                            "traffic": kernel_traffic("indexer_logits_kernel")},
        "topk_roofline": {"kernel": "indexer_topk_kernel", "bound": "hbm",
                          "achieved": topk_bytes / (t_avg * 1e-3) / 1e9, "unit": "GB/s", "peak": hbm_peak,
                          "frac": topk_bytes / (t_avg * 1e-3) / 1e9 / hbm_peak, "bytes_per_launch": topk_bytes,
                          "bytes": "the visible scores read once and the [M, 2048] int32 indices written once",
                          "traffic": kernel_traffic("indexer_topk_kernel")},
    }
    del logits_buf, topk_buf

    # ------------------------------------------ end to end through the C ABI
    # iq_prepare_q_host on page-locked host buffers: every step reads the
    # latent rows and positions from host memory and returns the FP4 codes and
    # scales to host memory, chunk by chunk, inside the timed region.
    h_lat = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_pos = torch.from_numpy(pos).pin_memory()
    h_q = torch.empty((M, N_Q // 2), dtype=torch.uint8).pin_memory()
    h_s = torch.empty((M, N_Q // 32), dtype=torch.uint8).pin_memory()
    work_h = torch.empty(iq.prepare_q_host_workspace_bytes(M), dtype=torch.uint8, device=dev)

    def e2e_step():
        iq.prepare_q_host(h_lat, w0, ws, h_pos, q_fp4=h_q, q_sf=h_s, workspace=work_h, stream=stream)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in eev:
        flush_l2()
        a.record(stream)
        e2e_step()
        b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in eev) / len(eev)
    clocks.__exit__(None, None, None)
    e2e = {"value": world * M / (e2e_ms * 1e-3), "unit": "tokens/s", "ms_per_step": e2e_ms,
           "call": "iq_prepare_q_host", "chunk_rows": iq.host_chunk_rows(),
           "h2d_bytes_per_step": h_lat.numel() * 2 + h_pos.numel() * 4,
           "d2h_bytes_per_step": h_q.numel() + h_s.numel()}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs = oracle_sample_seconds(ORACLE_SAMPLE_ROWS)
        cpu = {"value": ORACLE_SAMPLE_ROWS / secs, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"all {ORACLE_SAMPLE_ROWS} tokens of the prefill workload, FP64 numpy, "
                         f"one thread ({secs:.1f} s)",
               "cpu_model": host_cpu_model(), "host_cores": os.cpu_count()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3xe4m3->f32, e2m1 out", "data": "synthetic",
            "config": {"workload": "indexer-Q prefill chain: BF16 latent [4632, 1536] (N(0,1), 0.1% outliers x50) "
                                   "-> FP8 1x128 quantize -> block-scaled FP8 GEMM with W_q [8192, 1536] -> NeoX "
                                   "RoPE (positions 0..4631) -> Hadamard-128 -> MXFP4 [4632, 4096] + UE8M0 "
                                   "[4632, 256]",
                       "M": M, "K": K_LATENT, "N": N_Q, "parallelism": f"replicas x{world}",
                       "l2": "flushed between timed steps (256 MB write then 256 MB read), outside the event "
                             "intervals; back_to_back: rotating buffer sets over twice the L2 size"},
            "roofline": roofline, "quantizer": quantizer, "e2e": e2e, "cpu_baseline": cpu,
            "gpu_launches": 2 * args.steps,
            "clocks": clocks.summary(),
            "k1_chain_avg_ms": k1_avg_ms, "wall_s_timed": t_wall, "step_stats": step_stats,
            "back_to_back": back_to_back,
            "decode": decode, "sweep": sweep, "fp4_formats": fp4_formats, "indexer": indexer,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
