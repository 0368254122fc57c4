"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks, no GPU.

Multi-GPU runs of the benchmark are independent replicas (the work shards into
(request, KV head) units with no exchange), so the only cross-rank step is
taking the slowest rank's time and summing the units.
"""
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


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.5, 4.0][rank]
    worst = bench.max_over_ranks(ms)
    out[rank] = (worst, bench.replica_throughput(1000.0, worst * 1e-3, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1]
    worst, value = res[0]
    assert worst == 4.0
    assert value == pytest.approx(2 * 1000.0 / 4.0e-3)


def test_single_rank_identity():
    import bench
    assert bench.max_over_ranks(3.0) == 3.0
    assert bench.replica_throughput(10.0, 2.0, 1) == 5.0
