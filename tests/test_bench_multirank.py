"""The multi-rank bench aggregation on CPU: two gloo ranks, each timing its own replica.

bench.py runs one replica of the workload per rank (the path shards by
sequence with no exchange); the reported value is the bytes of all ranks over
the slowest rank's time.  This checks that host logic without a GPU.
"""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    my_ms = 1.0 + rank * 0.5                      # rank 1 is the slow one
    ms_max = bench.max_over_ranks(my_ms, "cpu")
    value = bench.job_throughput_gbs(10 ** 9, ms_max, world)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, ms_max, value))


def test_two_gloo_ranks_report_slowest_time_and_summed_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, value in out:
        assert ms_max == 1.5
        assert value == pytest.approx(2 * 1e9 / 1.5e-3 / 1e9)


def test_single_process_aggregation_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.job_throughput_gbs(2 * 10 ** 9, 1.0, 1) == pytest.approx(2000.0)
