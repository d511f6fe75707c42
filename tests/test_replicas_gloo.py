"""bench.py's whole-job figure for N replicas (one independent replica per rank,
no exchange step): world_size 2 over gloo on the CPU. Every rank must report the
slowest rank's time and the units of both ranks over it."""
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


def _rank(rank, ws, port, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    ms, rate = bench.replica_rate(0.05 * (rank + 1), 168, dist)   # rank 1 is the slow one
    q.put((rank, ms, rate))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate in got:
        assert ms == pytest.approx(0.10)                 # max over ranks
        assert rate == pytest.approx(2 * 168 / 0.10e-3)  # both ranks' nodes over it


def test_one_replica_is_its_own_rate():
    sys.path.insert(0, ROOT)
    import bench
    ms, rate = bench.replica_rate(0.064, 168)
    assert ms == 0.064 and rate == pytest.approx(168 / 0.064e-3)
