"""The N > 1 path of bench.py: replicas on every rank, no data exchange, whole-job
throughput = units of all ranks / the slowest rank's time. Run as two gloo ranks on CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r took (r + 1) seconds for its 10 units
    value, slowest = bench.combine_ranks(float(rank + 1), 10, dist, "cpu")
    out[rank] = (value, slowest)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_throughput_is_max_over_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        value, slowest = res[r]
        assert slowest == pytest.approx(2.0)
        assert value == pytest.approx(world * 10 / 2.0)


def test_single_process_needs_no_group():
    import bench

    assert bench.combine_ranks(0.5, 4) == (8.0, 0.5)
