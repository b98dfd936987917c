"""The multi-rank path of bench.py on CPU (gloo, two ranks): every rank runs
its own replica of the workload, so the job's time is the slowest rank's
and its throughput counts every rank's tokens.  Decode shards by sequence
with no exchange on the data path; the only collective is this timing
reduction."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seconds = [1.25, 2.5][rank]                 # rank 1 is the slower replica
        t = bench.max_over_ranks(seconds)
        q.put((rank, t, bench.job_throughput(world, 8, 100, t)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_two_ranks():
    import multiprocessing as mp
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
    for rank, t, v in got:
        assert t == 2.5                              # both ranks see the slowest replica's time
        assert v == pytest.approx(2 * 8 * 100 / 2.5)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0) == 3.0
    assert bench.job_throughput(1, 8, 10, 2.0) == 40.0
