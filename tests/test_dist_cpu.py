"""The multi-rank path of bench.py on CPU: two gloo ranks, no GPU.

Token batches are independent, so N GPUs run N replicas with no collective on
the data path; the only cross-rank steps are the barrier around the timed
region and the max over ranks of the elapsed time. Both are exercised here."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        elapsed = 0.5 * (rank + 1)  # rank 1 is the slow one
        t = bench.max_over_ranks(elapsed, world, device="cpu")
        out[rank] = bench.job_throughput(16, 100, world, t)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    out = mp.Manager().dict()
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    # 2 ranks x 16 tokens x 100 steps over the slowest rank's 1.0 s
    assert out[0] == out[1] == pytest.approx(3200.0)


def test_reference_arm_prints_only_on_rank_zero(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    import argparse

    ns = argparse.Namespace(gpus=2, steps=1, warmup=0, impl="reference", workload="tiny",
                            no_cpu_baseline=True, T=0, e2e_steps=0)
    bench.reference_arm(ns)
    assert capsys.readouterr().out == ""
