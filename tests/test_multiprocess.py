"""The N > 1 path of bench.py on CPU: world_size-2 gloo ranks, each a
replica with its own timing; the job time is the slowest rank's and the value
counts every rank's bytes (weak scaling, replicas only)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, ms, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        res = bench.replica_value(torch, ms[rank], world, 1_000_000, 10, "cpu")
        out[rank] = res
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    world = 2
    ms = [4.0, 5.0]
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), ms, out), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        max_ms, value = out[r]
        assert max_ms == 5.0
        # 2 replicas x 1 MB x 10 steps in 5 ms
        assert abs(value - 2 * 1e6 * 10 / 5e-3 / 1e9) < 1e-9


def test_single_process_value():
    ms, v = bench.replica_value(torch, 2.0, 1, 3_000_000, 4, "cpu")
    assert ms == 2.0 and abs(v - 3e6 * 4 / 2e-3 / 1e9) < 1e-12
