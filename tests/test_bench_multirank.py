"""bench.py's N > 1 timing path on two CPU ranks over gloo: every rank gets the maximum of
the ranks' times (the job ends when its slowest replica does), and the whole-job value is
the units all ranks processed divided by that time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = [7.0, 7.5][rank]                       # per-rank step time
        t = bench.reduce_max(dist, ms)
        dist.barrier()
        out.put((rank, t, bench.reduce_max(None, ms)))
    finally:
        dist.destroy_process_group()


def test_reduce_max_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [7.5, 7.5]          # both ranks see the slowest time
    assert [g[2] for g in got] == [7.0, 7.5]          # one process: the value itself
    flops_per_rank = 11.957e12
    value = flops_per_rank * 2 / (got[0][1] / 1e3) / 1e12
    assert value == pytest.approx(2 * 11.957 / 7.5e-3)
