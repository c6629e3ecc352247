"""Distributed-optimizer range maps: the oracle pinned by the page's toy and by element-wise
brute force, and the native engine bit-exact with the oracle (host-only)."""
import random

import pytest

from oracle import layout as L
from param_buffers_gb300 import abi, workloads as W

native = pytest.mark.skipif(not abi.LIB_PATH.exists(), reason="libgtp.so not built")


def toy_layout(golden):
    g = golden("toy_buffer.json")
    ps = [L.ParamSpec(n, k) for n, k in g["model_order"]]
    return g, L.compute_layout(ps, L.LayoutConfig(bucket_size=None, dp_size=2, use_distributed_optimizer=False))


def test_toy_ranges(golden):
    """[MLM] §6.3 / §9 Q5: WL's elements 0-10 belong to rank 0, element 11 to rank 1."""
    g, lay = toy_layout(golden)
    wl = [n for n, _ in g["model_order"]].index("WL")
    r0 = [r for r in L.shard_param_ranges(lay, 0, 2, 0) if r["param"] == wl]
    r1 = [r for r in L.shard_param_ranges(lay, 0, 2, 1) if r["param"] == wl]
    assert len(r0) == 1 and (r0[0]["param_start"], r0[0]["world_end"] - r0[0]["world_start"]) == (0, 11)
    assert len(r1) == 1 and (r1[0]["param_start"], r1[0]["world_end"] - r1[0]["world_start"]) == (11, 1)
    assert r1[0]["local_start"] == 0 and r0[0]["local_start"] == 0
    assert r1[0]["world_start"] == g["shard_boundary"]


def brute_owner(lay, buffer_id, dp):
    """element -> (rank, param) by walking every element of every bucket."""
    owner = {}
    for bid in lay.buffers[buffer_id].buckets:
        b = lay.buckets[bid]
        n = b.numel // dp
        for e in range(b.offset, b.offset + b.numel):
            rank = (e - b.offset) // n
            for pi in b.params:
                s, t = lay.param_index[pi][:2]
                if s <= e < t:
                    owner[e] = (rank, pi)
    return owner


@pytest.mark.parametrize("seed", range(25))
def test_ranges_cover_every_param_element_once(seed):
    rng = random.Random(seed)
    ps = [L.ParamSpec(f"p{i}", rng.choice([1, 5, 64, 100, 300, 999])) for i in range(rng.randint(1, 6))]
    dp = rng.choice([1, 2, 3, 4, 8])
    cfg = L.LayoutConfig(bucket_size=rng.choice([None, 200, 700]), dp_size=dp, use_distributed_optimizer=True)
    lay = L.compute_layout(ps, cfg)
    owner = brute_owner(lay, 0, dp)
    seen = {}
    for r in range(dp):
        for x in L.shard_param_ranges(lay, 0, dp, r):
            b = lay.buckets[x["bucket_id"]]
            s0 = b.offset + r * (b.numel // dp)
            assert x["bucket_start"] == x["world_start"] - b.offset
            assert x["local_start"] == x["world_start"] - s0
            assert x["param_start"] == x["world_start"] - lay.param_index[x["param"]][0]
            for e in range(x["world_start"], x["world_end"]):
                assert e not in seen
                seen[e] = (r, x["param"])
    assert seen == owner


@native
@pytest.mark.parametrize("seed", range(60))
def test_native_matches_oracle(seed):
    import param_buffers_gb300 as gtp
    rng = random.Random(500 + seed)
    sizes = [rng.choice([1, 7, 64, 65, 1000, 4096, 70_001]) for _ in range(rng.randint(1, 25))]
    dp = rng.choice([1, 2, 4, 8, 64])
    bs = rng.choice([None, 1000, 50_000])
    lay_o = L.compute_layout([L.ParamSpec(f"p{i}", n, is_expert_parallel=(i % 5 == 4)) for i, n in enumerate(sizes)],
                             L.LayoutConfig(bucket_size=bs, dp_size=dp))
    lay_n = gtp.gtp_buffer_layout([gtp.ParamDesc(n, is_expert_parallel=(i % 5 == 4)) for i, n in enumerate(sizes)],
                                  gtp.LayoutConfig(bucket_size=bs, dp_size=dp))
    for buf in range(len(lay_o.buffers)):
        for r in range(dp):
            assert gtp.gtp_shard_param_ranges(lay_n, buf, dp, r) == L.shard_param_ranges(lay_o, buf, dp, r)


@native
def test_native_7b_rank_ranges():
    import param_buffers_gb300 as gtp
    bw = W.seven_b_buffer()
    lay_n = gtp.gtp_buffer_layout([gtp.ParamDesc(p.numel, is_shared_embedding=p.is_shared_embedding)
                                   for p in bw.params], gtp.LayoutConfig(bw.bucket_size, 64))
    lay_o = L.compute_layout([L.ParamSpec(p.name, p.numel, is_shared_embedding=p.is_shared_embedding)
                              for p in bw.params], L.LayoutConfig(bw.bucket_size, 64))
    for r in (0, 17, 63):
        got = gtp.gtp_shard_param_ranges(lay_n, 0, 64, r)
        assert got == L.shard_param_ranges(lay_o, 0, 64, r)
        # [BUF] §8: each rank owns 1M elements of every full bucket
        full = [x for x in got if lay_n.buckets[x["bucket_id"]]["numel"] == 64_000_000]
        per_bucket = {}
        for x in full:
            per_bucket[x["bucket_id"]] = per_bucket.get(x["bucket_id"], 0) + x["world_end"] - x["world_start"]
        assert set(per_bucket.values()) == {1_000_000}


@native
def test_native_errors():
    import ctypes as C
    lib = abi.load()
    idx = (abi.gtp_param_index * 1)(abi.gtp_param_index(0, 10, 0, 10, 0, 0))
    bk = (abi.gtp_bucket_desc * 1)(abi.gtp_bucket_desc(0, 10, 10, 0, 1))
    n = C.c_int32(0)
    assert lib.gtp_shard_param_ranges(idx, 1, bk, 1, 0, 4, 0, None, C.byref(n)) == abi.GTP_E_SHAPE   # 10 % 4
    assert lib.gtp_shard_param_ranges(idx, 1, bk, 1, 0, 2, 2, None, C.byref(n)) == abi.GTP_E_ARG     # rank >= dp
    assert lib.gtp_shard_param_ranges(idx, 1, bk, 1, 0, 2, 1, None, C.byref(n)) == abi.GTP_OK and n.value == 1
