"""Replica timing across ranks (no GPU): two gloo ranks on the CPU run the
same max-over-ranks reduction and whole-job throughput the benchmark uses."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank  # rank 1 is the straggler
    ms = bench.max_over_ranks(local_ms, "cpu", world)
    q.put((rank, ms, bench.job_throughput(1e12, world, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, tput in res:
        assert ms == 15.0
        assert tput == pytest.approx(2 * 1e12 / 15e-3 / 1e12)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, "cpu", 1) == 3.5
    assert bench.job_throughput(2e12, 1, 1000.0) == pytest.approx(2.0)
