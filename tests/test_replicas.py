"""The multi-GPU path is replicas only: each rank runs the whole workload on
its own GPU, and bench.py's only collectives are a barrier and the
max-over-ranks of the timed seconds.  These tests run that host-side logic as
two gloo ranks on the CPU.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, seconds, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    got_rank, got_world, got_local = bench.dist_env()
    dist.init_process_group("gloo", rank=got_rank, world_size=got_world)
    try:
        bench._barrier(got_world)
        worst = bench._max_over_ranks(seconds[rank], got_world, "cpu")
        bench._barrier(got_world)
        out[rank] = (got_rank, got_world, got_local, worst)
    finally:
        dist.destroy_process_group()


def test_two_replicas_share_the_slowest_time():
    world = 2
    seconds = [0.125, 0.5]
    ctx = mp.get_context("spawn")
    with ctx.Manager() as manager:
        out = manager.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), seconds, out), nprocs=world,
                           join=True, start_method="spawn")
        results = dict(out)
    assert sorted(results) == [0, 1]
    for rank, (r, w, local, worst) in results.items():
        assert (r, w, local) == (rank, world, rank)
        assert worst == max(seconds)        # every rank reports the job's slowest replica


def test_single_process_needs_no_collective(monkeypatch):
    for name in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(name, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench._max_over_ranks(0.25, 1, "cpu") == 0.25
    bench._barrier(1)                        # no process group: nothing to wait for
    assert not dist.is_initialized()
