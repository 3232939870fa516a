"""The multi-rank path of bench.py on the CPU: world_size-2 `gloo` process groups (the step
itself has no exchange; ranks are independent replicas and only the timing is combined)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(dist, values[rank])
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world = 2
    values = [[140.0, 150.5], [141.5, 149.0]]  # per-rank (device ms/step, end-to-end ms/step)
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, values, out), nprocs=world, join=True)
    for r in range(world):
        assert out[r] == [141.5, 150.5]  # every rank sees the slowest rank's times


def test_job_throughput_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, [3, 4]) == [3.0, 4.0]  # single process: unchanged
    one = bench.job_tokens_per_s(1, 512, 140.0)
    assert abs(one - 512 / 0.140) < 1e-9
    # weak scaling: per-rank work fixed, whole-job tokens add up over the ranks
    assert abs(bench.job_tokens_per_s(4, 512, 140.0) - 4 * one) < 1e-9
