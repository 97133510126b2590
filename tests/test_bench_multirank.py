"""The multi-rank host logic of bench.py on CPU: two gloo ranks (world size 2) each time
their own replica; the job reports the slowest rank's step time and all ranks' tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        local_ms = [0.25, 0.40][rank]  # rank 1 is the slower replica
        bench.barrier(world)
        ms_max, value = bench.aggregate(local_ms, 32, world, torch.device("cpu"))
        results[rank] = (ms_max, value)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregate_takes_slowest_rank_and_all_tokens():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.start_processes(_rank, args=(world, port, results), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(results)
    for r in range(world):
        ms_max, value = res[r]
        assert ms_max == pytest.approx(0.40)
        assert value == pytest.approx(world * 32 / 0.40e-3)


def test_single_rank_aggregate_is_local():
    ms_max, value = bench.aggregate(0.5, 10, 1, torch.device("cpu"))
    assert ms_max == 0.5 and value == pytest.approx(10 / 0.5e-3)
