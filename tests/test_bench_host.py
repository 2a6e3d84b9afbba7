"""Host logic of bench.py's multi-process path (one replica per GPU under torchrun):
the whole-job time is the slowest rank's. Two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, values, out):
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank], dist, "cpu")
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        values = [0.25, 0.75]
        mp.start_processes(_rank, args=(2, _free_port(), values, out), nprocs=2, join=True,
                           start_method="spawn")
        assert dict(out) == {0: 0.75, 1: 0.75}


def test_max_over_ranks_single_process():
    import bench
    assert bench.max_over_ranks(1.5) == 1.5


if __name__ == "__main__":
    pytest.main([__file__])
