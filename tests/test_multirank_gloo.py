"""Two CPU ranks over gloo: the ZeRO-1 loop of [MLM] §6.4 / [BUF] §6.5 on the toy buffer
and on a bucketed layout from the native layout engine.

Each rank accumulates its own microbatch gradients into its flat grad buffer; the bucket
is summed across ranks and each rank keeps its dp shard (reduce-scatter, done as
all_reduce + slice since gloo has no reduce_scatter), scales it by 1/dp, runs AdamW on
its shard of the fp32 master / m / v (the oracle's arithmetic; no GPU here), casts to
bf16 and all-gathers the bf16 shards.  The result must equal single-process AdamW on the
dp-averaged gradient - exactly, since the update is elementwise (the page's toy reports
"max diff < 0.01" and "two steps equal: True").
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import adamw as A
from oracle import floats as F
from oracle import layout as L

H = A.AdamWHparams()


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def local_grads(rank: int, numel: int, step: int) -> np.ndarray:
    g = torch.Generator().manual_seed(100 * step + rank)
    return (torch.randn(numel, generator=g) * 1e-3).numpy().astype(np.float32)


def zero1_steps(rank, world, numel, buckets, master0, steps):
    """Returns this rank's view of param_data (bf16 bits) after `steps` ZeRO-1 steps."""
    master = master0.copy().astype(np.float64)
    m = np.zeros(numel)
    v = np.zeros(numel)
    param = F.f32_to_bf16_bits(master0.astype(np.float32))
    for t in range(1, steps + 1):
        grad = torch.from_numpy(local_grads(rank, numel, t))
        for b in buckets:
            view = grad[b.offset:b.offset + b.numel]
            dist.all_reduce(view)                                  # sum over dp ranks
        for b in buckets:
            lo, hi = L.shard_ranges(b, world)[rank]
            g = A.scale_grad(grad.numpy()[lo:hi], np.full(hi - lo, 1.0 / world)).astype(np.float64)
            master[lo:hi], m[lo:hi], v[lo:hi] = A.adamw(master[lo:hi], g, m[lo:hi], v[lo:hi], t, H)
            # bf16 bit patterns travel as int32 (gloo has no 16-bit integer collectives)
            mine = torch.from_numpy(F.f32_to_bf16_bits(master[lo:hi].astype(np.float32)).astype(np.int32))
            parts = [torch.empty_like(mine) for _ in range(world)]
            dist.all_gather(parts, mine)                           # param all-gather
            param[b.offset:b.offset + b.numel] = torch.cat(parts).numpy().astype(np.uint16)
    return param


def worker(rank, world, port, numel, bucket_specs, master0, steps, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        buckets = [L.Bucket(0, o, n, n) for o, n in bucket_specs]
        out[rank] = zero1_steps(rank, world, numel, buckets, master0, steps)
    finally:
        dist.destroy_process_group()


def single_process(world, numel, master0, steps):
    master = master0.astype(np.float64)
    m = np.zeros(numel)
    v = np.zeros(numel)
    for t in range(1, steps + 1):
        tot = sum(local_grads(r, numel, t).astype(np.float32) for r in range(world))   # fp32 sum, 2 ranks: exact order
        g = A.scale_grad(tot.astype(np.float32), np.full(numel, 1.0 / world)).astype(np.float64)
        master, m, v = A.adamw(master, g, m, v, t, H)
    return F.f32_to_bf16_bits(master.astype(np.float32))


def run(numel, bucket_specs, steps=2, world=2):
    master0 = (torch.randn(numel, generator=torch.Generator().manual_seed(7)) * 0.02).numpy().astype(np.float32)
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(worker, args=(world, free_port(), numel, bucket_specs, master0, steps, out),
                           nprocs=world, join=True, start_method="spawn")
        results = [out[r] for r in range(world)]
    ref = single_process(world, numel, master0, steps)
    for r in results:
        assert np.array_equal(r, results[0])                         # all ranks hold the same params
    diff = np.abs(F.bf16_bits_to_f64(results[0]) - F.bf16_bits_to_f64(ref)).max()
    return diff, np.array_equal(results[0], ref)


def test_toy_buffer_two_ranks(golden):
    """[MLM] §6.3/§6.4 toy: numel 22, one bucket, shard boundary 11, two steps."""
    g = golden("toy_buffer.json")
    lay = L.compute_layout([L.ParamSpec(n, k) for n, k in g["model_order"]],
                           L.LayoutConfig(bucket_size=None, dp_size=2, use_distributed_optimizer=False))
    specs = [(b.offset, b.numel) for b in lay.buckets]
    assert L.shard_ranges(lay.buckets[0], 2)[0][1] == g["shard_boundary"]
    diff, equal = run(lay.buffers[0].numel, specs, steps=2)
    assert diff < g["adam_parity_max_diff_below"]
    assert equal == g["two_step_parity"]


def test_bucketed_distopt_layout_two_ranks():
    """A padded, multi-bucket dist-opt layout from the native engine (host-only)."""
    from param_buffers_gb300 import abi
    if not abi.LIB_PATH.exists():
        pytest.skip("libgtp.so not built")
    import param_buffers_gb300 as gtp
    params = [gtp.ParamDesc(n) for n in (300, 77, 1000, 5, 640, 129)]
    lay = gtp.gtp_buffer_layout(params, gtp.LayoutConfig(bucket_size=700, dp_size=2))
    assert len(lay.buckets) > 1 and all(b["numel"] % 2 == 0 for b in lay.buckets)
    specs = [(b["offset"], b["numel"]) for b in lay.buckets]
    diff, equal = run(lay.buffers[0]["numel"], specs, steps=3)
    assert equal and diff == 0.0
