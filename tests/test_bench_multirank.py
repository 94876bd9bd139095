"""The multi-GPU form of bench.py runs one replica of the workload per rank
(the product needs no exchange) and reports the whole job's throughput over
the slowest rank's time.  Checked here with two gloo ranks on the CPU."""
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


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [10.0, 25.0][rank]          # rank 1 is the slow one
    value, max_ms = bench.aggregate_throughput(local_ms, flops_per_step=1e12, steps=5, dist=dist)
    out[rank] = (value, max_ms)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        value, max_ms = out[r]
        assert max_ms == 25.0
        assert value == pytest.approx(world * 1e12 * 5 / 25e-3 / 1e12)


def test_single_process_is_its_own_time():
    sys.path.insert(0, ROOT)
    import bench
    value, max_ms = bench.aggregate_throughput(4.0, 2e12, 3, dist=None)
    assert max_ms == 4.0 and value == pytest.approx(2e12 * 3 / 4e-3 / 1e12)
