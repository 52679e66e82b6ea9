"""Replicas-only scaling of bench.py: with N ranks (gloo on CPU, world size
2) the step time is the maximum over ranks and every rank's rows count."""

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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    assert bench._dist() == (world, rank)
    ms = bench.aggregate_ms(10.0 + 5.0 * rank, dist, torch.device("cpu"))
    out[rank] = ms
    dist.barrier()
    dist.destroy_process_group()


def test_step_time_is_max_over_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == 15.0
    # value = all ranks' rows / max step time (weak scaling of independent replicas)
    rows = 8192
    assert world * rows / (out[0] / 1e3) == pytest.approx(2 * 8192 / 0.015)
