"""reduce_scatter_with_fp32_accumulation on CPU ranks over gloo ([BUF] §9.1): every rank
sends each dp rank that rank's slice of its bf16 grad bucket with one all-to-all, then
adds the world_size slices it received in fp32, in rank order (the oracle's local sum,
R20), and casts to bf16.  Checked: the all-to-all delivers the slices in rank order (each
rank's shard equals the local sum of the buckets' slices taken directly), the result is
the fp32 sum of the ranks' values within the recursive-summation bound, and the shards of
all ranks concatenate to the whole bucket's reduction."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import floats as F
from oracle import rs_sum as R


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def bucket_of(rank: int, n: int) -> np.ndarray:
    g = torch.Generator().manual_seed(1000 + rank)
    x = torch.randn(n, generator=g) * torch.exp2(torch.randint(-10, 10, (n,), generator=g).float())
    return F.f32_to_bf16_bits(x.numpy())


def _rank(rank, world, n, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # bf16 bit patterns travel as int32 (gloo has no 16-bit integer collectives)
        mine = torch.from_numpy(bucket_of(rank, n).astype(np.int32))
        recv = torch.empty_like(mine)
        dist.all_to_all_single(recv, mine)          # slice k of my bucket to rank k; rank j's slice r to me
        s = n // world
        got = recv.numpy().astype(np.uint16).reshape(world, s)
        out.put((rank, R.local_sum([got[j] for j in range(world)], out_bf16=True)))
    finally:
        dist.destroy_process_group()


def run(world: int, n: int) -> dict:
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, n, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    shards = dict(q.get(timeout=60) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return shards


def test_a2a_reduce_scatter_with_fp32_accumulation():
    world, n = 4, 4096
    shards = run(world, n)
    buckets = [bucket_of(r, n) for r in range(world)]
    s = n // world
    for r in range(world):
        direct = R.local_sum([b[r * s:(r + 1) * s] for b in buckets], out_bf16=True)
        assert np.array_equal(shards[r], direct)                     # slices arrive in rank order
        f32 = R.local_sum_fp32([b[r * s:(r + 1) * s] for b in buckets]).astype(np.float64)
        exact = np.sum([F.bf16_bits_to_f64(b[r * s:(r + 1) * s]) for b in buckets], axis=0)
        assert np.all(np.abs(f32 - exact) <= R.sum_bound([b[r * s:(r + 1) * s] for b in buckets]))
    whole = np.concatenate([shards[r] for r in range(world)])
    assert np.array_equal(whole, R.local_sum(buckets, out_bf16=True))  # the bucket's reduction, sharded
