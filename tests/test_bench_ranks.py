"""The multi-GPU bookkeeping of bench.py, on CPU: two gloo ranks over 127.0.0.1.

bench.py --gpus N runs one replica of the workload per rank (weak scaling, no data-path collective); the
only cross-rank steps are the barriers around the timed region and the maximum of the timed interval over
the ranks, from which the whole-job rate is formed. The reference arm runs on rank 0 alone.
"""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")     # rank 1 is the slower one
        out[rank] = (ms, bench.job_rate(world, 100.0, ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_rate():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, rate = res[0]
    assert ms == 15.0
    assert rate == pytest.approx(2 * 100.0 / 0.015)


def test_single_process_keeps_its_own_time():
    assert bench.max_over_ranks(12.5, "cpu") == 12.5
    assert bench.job_rate(1, 50.0, 10.0) == pytest.approx(5000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        gpus, steps, warmup = 2, 1, 0

    w = wl.WORKLOADS["tiny48"]
    assert bench.run_reference(Args, w) == 0
    assert capsys.readouterr().out == ""
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("LOCAL_RANK", "0")
    assert bench.run_reference(Args, w) == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["n_gpus"] == 2
