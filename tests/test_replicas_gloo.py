"""The multi-GPU mode of the benchmark runs independent replicas (the path has no
exchange step); its only cross-rank logic is the barrier and the max of the
replicas' times.  Checked here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from tests.conftest import ROOT


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed_ms = 10.0 + 5.0 * rank           # rank 1 is the slow replica
    dist.barrier()
    m = bench.reduce_max_over_ranks(elapsed_ms, world, "cpu")
    us = bench.aggregate_us_per_unit(m, units_per_rank=16 * 20, world=world)
    q.put((rank, m, us))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, us in res:
        assert m == 15.0
        assert us == pytest.approx(15.0 * 1e3 / (16 * 20 * 2))
