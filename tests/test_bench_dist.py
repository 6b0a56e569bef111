"""The N > 1 path of bench.py on CPU: two gloo ranks agree on the slowest
rank's time, and the whole-job value counts every rank's tokens."""
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


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [0.30, 0.45][rank]
        slowest = bench.max_over_ranks(local_ms)
        results[rank] = (slowest, bench.weak_scaling_value(1984, world, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_sum_tokens():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
        got = dict(results)
    for rank in range(world):
        slowest, value = got[rank]
        assert slowest == pytest.approx(0.45)
        assert value == pytest.approx(2 * 1984 / 0.45e-3)


def test_single_process_needs_no_process_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(0.3) == 0.3
    assert bench.weak_scaling_value(1984, 1, 0.5) == pytest.approx(1984 / 0.5e-3)
