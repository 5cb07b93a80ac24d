"""The multi-GPU mode of bench.py is replicas only (a decode step is one dependency
chain; nothing is exchanged between GPUs). This checks its host logic on CPU with
two gloo ranks: the job's time is the slowest rank's, and the throughput counts
every replica's bytes."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    total_ms, e2e_s = bench.slowest_replica(10.0 + 5.0 * rank, 0.5 - 0.1 * rank, world, torch.device("cpu"))
    out[rank] = (total_ms, e2e_s)
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == (15.0, 0.5)


def test_replica_throughput_counts_every_rank():
    import bench
    one = bench.replicas_gbs(669_901_824, 1, 0.8)
    assert bench.replicas_gbs(669_901_824, 4, 0.8) == pytest.approx(4 * one)
    assert one == pytest.approx(669_901_824 / 0.8e-3 / 1e9)
    assert bench.slowest_replica(3.0, 1.0, 1, None) == (3.0, 1.0)
