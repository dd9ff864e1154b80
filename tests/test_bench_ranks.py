"""The multi-process path of bench.py on the CPU: two ranks over gloo (as
torchrun would start them, rendezvous on 127.0.0.1) agree on the slowest
rank's times, which the whole-job throughput divides by."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: a step time of 10 + r ms and a verify time of 5 - r ms
        out[rank] = bench.max_over_ranks([10.0 + rank, 5.0 - rank], "cpu")
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_times_are_the_maximum_over_two_ranks():
    if not torch.distributed.is_available() or not torch.distributed.is_gloo_available():
        pytest.skip("torch.distributed with gloo is not available")
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        got = dict(out)
    assert got[0] == [11.0, 5.0]
    assert got[1] == [11.0, 5.0]


def test_single_process_returns_its_own_times():
    assert bench.max_over_ranks([3.0, 4.0], "cpu") == [3.0, 4.0]
