"""Host logic of the replica mode (bench.py under torchrun): every rank times its
own replica, the slowest rank's time is shared by an all-reduce MAX, and the
whole-job rate sums the ranks' work.  Runs as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [3.0, 5.0][rank]
    ms = bench.max_over_ranks(local_ms, dist, "cpu")
    rate = bench.whole_job_rate(1.0e12, world, ms)
    q.put((rank, ms, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_share_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, rate in got:
        assert ms == pytest.approx(5.0)
        assert rate == pytest.approx(2 * 1.0e12 / 5.0e-3)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(4.0) == 4.0
    assert bench.whole_job_rate(2.0, 1, 1000.0) == pytest.approx(2.0)
