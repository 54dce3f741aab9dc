"""Host logic of the multi-GPU bench path on CPU: replicas only (the path has
no exchange step), so the only cross-rank step is the timing reduction --
the slowest rank's step time, and the whole-job rate of all ranks' units
over it.  Two gloo ranks on 127.0.0.1."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        my_ms = [0.25, 0.75][rank]
        ms = bench.max_over_ranks(my_ms, world)
        out[rank] = (ms, bench.whole_job_rate(4632, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_time():
    port = _free_port()
    with mp.Manager() as manager:
        out = manager.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        got = dict(out)
    assert got[0][0] == pytest.approx(0.75) and got[1][0] == pytest.approx(0.75)
    assert got[0][1] == pytest.approx(2 * 4632 / 0.75e-3)
    assert got[0] == got[1]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.whole_job_rate(100, 1, 2.0) == pytest.approx(50000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup, gpus = 1, 0, 2
    assert bench.run_reference(Args()) is None
    assert capsys.readouterr().out == ""
