"""Host logic of the multi-replica benchmark, on CPU with gloo (world size 2).

The layer forward has no exchange step, so N GPUs run N independent replicas;
the job time is the slowest replica's and the throughput counts every
replica's tokens.  These tests run that reduction across two real processes.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, local_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(local_ms[rank], world)
        out[rank] = (ms, bench.job_tokens_per_s(world, 4096, 20, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_two_ranks():
    world, port = 2, _free_port()
    local_ms = [40.0, 43.5]  # rank 1 is the slow replica
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, local_ms, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1]  # every rank sees the same job time
    ms, value = res[0]
    assert ms == 43.5
    assert value == pytest.approx(2 * 4096 * 20 / 0.0435)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.job_tokens_per_s(1, 512, 10, 5.0) == pytest.approx(512 * 10 / 0.005)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun the other ranks exit without work and print nothing."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload, T, alpha, experts, activation = "mixtral", None, None, None, None
        steps, warmup, gpus = 1, 3, 2

    assert bench.run_reference(Args()) is None
    assert capsys.readouterr().out == ""
