"""Pins of the layout oracle: page-printed layouts and counts, invariants, brute force."""
import math
import random

import pytest

from oracle import layout as L
from param_buffers_gb300 import workloads as W


def specs(params):
    return [L.ParamSpec(p.name, p.numel, p.dtype, is_shared_embedding=p.is_shared_embedding) for p in params]


def cfg_of(bw: W.BufferWorkload) -> L.LayoutConfig:
    return L.LayoutConfig(bucket_size=bw.bucket_size, dp_size=bw.dp_size,
                          use_distributed_optimizer=bw.use_distributed_optimizer,
                          pad_buckets_for_high_nccl_busbw=bw.pad_buckets_for_high_nccl_busbw)


# ----------------------------------------------------------------------------- page pins

def test_toy_buffer_default_layout(golden):
    """[MLM] §6.3 toy: W1(6), W2(4), WL(12) -> WL [0,12) W2 [12,16) W1 [16,22), numel 22, pad 0."""
    g = golden("toy_buffer.json")
    ps = [L.ParamSpec(n, k) for n, k in g["model_order"]]
    lay = L.compute_layout(ps, L.LayoutConfig(bucket_size=None, dp_size=g["dp_size"],
                                              use_distributed_optimizer=False))
    names = [n for n, _ in g["model_order"]]
    for i, n in enumerate(names):
        s, e, b, buf = lay.param_index[i]
        assert [s, e] == g["ranges"][n]
    assert lay.buffers[0].numel == g["numel"]
    bk = lay.buckets[0]
    assert bk.numel - bk.numel_unpadded == g["pad"]
    shards = L.shard_ranges(bk, g["dp_size"])
    assert shards[0][1] == g["shard_boundary"]
    wl = lay.param_index[names.index("WL")]
    assert (wl[0], shards[0][1] - 1) == tuple(g["wl_rank0_elements"])
    assert (shards[1][0], wl[1] - 1) == tuple(g["wl_rank1_elements"])


def test_toy_is_not_the_distopt_layout(golden):
    """With 64-element start padding W2 would start at 64, not 12: the toy is the default layout."""
    g = golden("toy_buffer.json")
    ps = [L.ParamSpec(n, k) for n, k in g["model_order"]]
    lay = L.compute_layout(ps, L.LayoutConfig(bucket_size=None, dp_size=2, use_distributed_optimizer=True))
    assert lay.param_index[1][0] == 64
    assert lay.buffers[0].numel != g["numel"]


def test_7b_bucket_count_and_ledger(golden):
    """[BUF] §8: 64M buckets, 29 full + 1 tail + 1 for the tied embedding; the memory ledger."""
    g = golden("ledger_7b.json")
    bw = W.seven_b_buffer()
    assert bw.bucket_size == g["bucket_size_elements"] == L.default_bucket_size(g["dp"])
    total = sum(p.numel for p in bw.params)
    assert total == g["P_per_rank"] == g["P"] / (g["tp"] * g["pp"])
    lay = L.compute_layout(specs(bw.params), cfg_of(bw))
    nb = lay.buckets
    full = [b for b in nb if b.numel_unpadded == g["bucket_size_elements"]]
    assert len(full) == g["full_buckets"]
    assert len(nb) == g["full_buckets"] + g["tail_buckets"] + g["extra_bucket_if_tied_embedding"]
    emb_bucket = lay.param_index[0][2]
    assert lay.buckets[emb_bucket].params == [0]            # tied embedding alone
    assert emb_bucket == len(nb) - 1                        # model head = end of the buffer
    numel = lay.buffers[0].numel
    assert round(numel * 4 / 1e9, 2) == g["grad_data_GB"]
    assert round(numel * 2 / 1e9, 2) == g["param_data_GB"]
    assert round(12 * numel / g["dp"] / 1e9, 2) == g["master_m_v_sharded_GB_approx"]
    assert round(12 * numel / 1e9, 1) == g["master_m_v_unsharded_GB"]
    b0 = nb[0]
    assert b0.numel // g["dp"] == g["per_rank_shard_elements"]
    assert b0.numel * 4 / 1e6 == g["rs_per_bucket_MB"]
    assert round(numel * 4 * (g["dp"] - 1) / g["dp"] / 1e9, 1) == g["grad_rs_per_iter_GB_approx"]
    assert round(numel * 2 * (g["dp"] - 1) / g["dp"] / 1e9, 1) == g["param_ag_per_iter_GB_approx"]


def test_7b_busbw_padding_bound(golden):
    """[BUF] §8: busbw padding costs at most about 29 x (2^16 - 1) elements (~1.9M, ~7.6 MB)."""
    g = golden("ledger_7b.json")
    bw = W.seven_b_buffer(busbw=True)
    lay = L.compute_layout(specs(bw.params), cfg_of(bw))
    pads = [b.numel - b.numel_unpadded for b in lay.buckets]
    assert all(0 <= p <= 2 ** 16 - 1 for p in pads)
    assert all(b.numel % math.lcm(64, 128, 2 ** 16) == 0 for b in lay.buckets)
    total_pad = sum(pads)
    assert total_pad <= g["full_buckets"] * (2 ** 16 - 1)
    assert round(g["full_buckets"] * (2 ** 16 - 1) / 1e5) * 1e5 == g["busbw_padding_bound_elements_approx"]
    assert round(g["full_buckets"] * (2 ** 16 - 1) * 4 / 1e6, 1) == g["busbw_padding_bound_MB_approx"]


def test_default_bucket_size_rule():
    """[BUF] §4.3: max(40M, 1M x dp) elements; the num_buckets variant."""
    assert L.default_bucket_size(2) == 40_000_000
    assert L.default_bucket_size(64) == 64_000_000
    assert L.bucket_size_for_num_buckets(1000, 3) == 333


# ----------------------------------------------------------------------------- derived values

def test_workload_layouts():
    t = L.compute_layout(specs(W.tiny_buffer().params), cfg_of(W.tiny_buffer()))
    assert [t.param_index[i][:2] for i in range(2)] == [(512, 131584), (0, 512)]
    assert len(t.buckets) == 1 and t.buffers[0].numel == 131584
    lay = L.compute_layout(specs(W.layer_buffer().params), cfg_of(W.layer_buffer()))
    assert len(lay.buckets) == 1 and lay.buffers[0].numel == 30_412_800
    names = [p.name for p in W.layer_buffer().params]
    got = {n: lay.param_index[i][:2] for i, n in enumerate(names)}
    assert got["fc2"] == (0, 8388608) and got["fc1"] == (8388608, 25165824)
    assert got["proj"] == (25167872, 27265024) and got["qkv"] == (27265024, 30410752)
    st = L.compute_layout(specs(W.stage_buffer().params), cfg_of(W.stage_buffer()))
    assert st.buffers[0].numel == 374_636_544 and len(st.buckets) == 6
    assert sum(b.numel - b.numel_unpadded for b in st.buckets) == 0
    sb = L.compute_layout(specs(W.seven_b_buffer().params), cfg_of(W.seven_b_buffer()))
    assert sb.buffers[0].numel == 1_875_000_064 and len(sb.buckets) == 31
    bb = L.compute_layout(specs(W.seven_b_buffer(True).params), cfg_of(W.seven_b_buffer(True)))
    assert bb.buffers[0].numel == 1_875_902_464 and len(bb.buckets) == 31
    real = W.seven_b_realistic_params()
    assert sum(p.numel for p in real) == 1_864_863_744
    rl = L.compute_layout(specs(real), L.LayoutConfig(bucket_size=64_000_000, dp_size=64))
    assert len(rl.buckets) == 26


# ----------------------------------------------------------------------------- invariants

def check_invariants(params, cfg, lay):
    div = L.bucket_end_divisor(cfg) if cfg.use_distributed_optimizer else 1
    for bi, buf in enumerate(lay.buffers):
        bks = [lay.buckets[k] for k in buf.buckets]
        # buckets tile [0, numel) contiguously
        pos = 0
        for b in bks:
            assert b.offset == pos and b.numel >= b.numel_unpadded > 0
            pos += b.numel
            if cfg.use_distributed_optimizer:
                assert b.numel % div == 0 and b.numel % cfg.dp_size == 0
                assert b.numel - b.numel_unpadded < div
            else:
                assert b.numel == b.numel_unpadded
        assert pos == buf.numel
        # params: reverse model order, aligned, inside their bucket, no overlap
        members = buf.params
        starts = [lay.param_index[i][0] for i in reversed(members)]
        assert starts == sorted(starts)
        prev_end = 0
        for i in reversed(members):
            s, e, b, bid = lay.param_index[i]
            assert bid == bi and e - s == params[i].numel and s >= prev_end
            if cfg.use_distributed_optimizer:
                assert s % 64 == 0
            else:
                assert s == prev_end
            bk = lay.buckets[b]
            assert bk.offset <= s and e <= bk.offset + bk.numel_unpadded
            assert bk.param_to_index[i] == (s - bk.offset, e - bk.offset)
            prev_end = e
        # a bucket is closed exactly when it reaches bucket_size (or before a shared embedding)
        for b in bks:
            last = max(b.params, key=lambda i: lay.param_index[i][1])
            grown = lay.param_index[last][1] - b.offset
            if cfg.bucket_size is not None:
                for i in b.params:
                    if i != last:
                        assert lay.param_index[i][1] - b.offset < cfg.bucket_size
        sizes = sum(params[i].numel for i in members)
        gaps = sum(b.numel_unpadded for b in bks) - sizes
        assert gaps >= 0 and (gaps == 0 or cfg.use_distributed_optimizer)


def brute_force_layout(params, cfg):
    """Element-at-a-time restatement of the rules (tiny lists only)."""
    out = {}
    buckets = []
    keys = []
    for i, p in enumerate(params):
        k = L.buffer_key(p, cfg)
        if k not in keys:
            keys.append(k)
    for k in keys:
        members = [i for i, p in enumerate(params) if L.buffer_key(p, cfg) == k]
        cur, bstart, open_ = 0, 0, []

        def close():
            nonlocal cur, bstart, open_
            unpadded = cur - bstart
            if cfg.use_distributed_optimizer:
                while cur % cfg.dp_size or cur % 128 or (cfg.pad_buckets_for_high_nccl_busbw and cur % 65536):
                    cur += 1
            buckets.append((bstart, unpadded, cur - bstart, list(open_)))
            bstart, open_ = cur, []

        for i in reversed(members):
            p = params[i]
            iso = cfg.use_distributed_optimizer and p.is_shared_embedding
            if iso and open_:
                close()
            if cfg.use_distributed_optimizer:
                while cur % 64:
                    cur += 1
            s = cur
            for _ in range(p.numel):
                cur += 1
            out[i] = (s, cur)
            open_.append(i)
            if iso or (cfg.bucket_size is not None and cur - bstart >= cfg.bucket_size):
                close()
        if open_:
            close()
    return out, buckets


@pytest.mark.parametrize("seed", range(40))
def test_random_lists_against_brute_force(seed):
    rng = random.Random(seed)
    n = rng.randint(1, 7)
    ps = []
    for i in range(n):
        ps.append(L.ParamSpec(f"p{i}", rng.choice([1, 3, 31, 64, 65, 100, 127, 200, 700]),
                              dtype=rng.choice(["bf16", "bf16", "fp32"]),
                              is_expert_parallel=rng.random() < 0.2,
                              is_shared_embedding=(i == 0 and rng.random() < 0.5)))
    cfg = L.LayoutConfig(bucket_size=rng.choice([None, 50, 128, 300, 1000]), dp_size=rng.choice([1, 2, 3, 8]),
                         use_distributed_optimizer=rng.random() < 0.7,
                         pad_buckets_for_high_nccl_busbw=rng.random() < 0.2,
                         grad_reduce_in_fp32=rng.random() < 0.8)
    lay = L.compute_layout(ps, cfg)
    check_invariants(ps, cfg, lay)
    ref, ref_buckets = brute_force_layout(ps, cfg)
    for i in range(n):
        assert lay.param_index[i][:2] == ref[i]
    got = [(b.offset, b.numel_unpadded, b.numel, b.params) for b in lay.buckets]
    assert got == ref_buckets


def test_invariants_on_workloads():
    for bw in (W.tiny_buffer(), W.layer_buffer(), W.stage_buffer(), W.seven_b_buffer(), W.seven_b_buffer(True)):
        ps = specs(bw.params)
        check_invariants(ps, cfg_of(bw), L.compute_layout(ps, cfg_of(bw)))


def test_buffer_key_grouping():
    """[BUF] §3: one buffer per key, keys in first-appearance order; uint8 storage key for FP8."""
    ps = [L.ParamSpec("a", 10, "bf16"), L.ParamSpec("e", 10, "bf16", is_expert_parallel=True),
          L.ParamSpec("q", 10, "bf16", quantized_storage=True), L.ParamSpec("b", 10, "bf16")]
    cfg = L.LayoutConfig(bucket_size=None, dp_size=1, grad_reduce_in_fp32=False)
    lay = L.compute_layout(ps, cfg)
    assert [b.key for b in lay.buffers] == [
        L.BufferKey("bf16", "bf16", False, False), L.BufferKey("bf16", "bf16", True, False),
        L.BufferKey("uint8", "bf16", False, False)]
    assert lay.buffers[0].params == [0, 3]
    assert lay.param_index[3][:2] == (0, 10) and lay.param_index[0][:2] == (64, 74)
    lay32 = L.compute_layout(ps, L.LayoutConfig(bucket_size=None, grad_reduce_in_fp32=True))
    assert all(b.key.grad_dtype == "fp32" for b in lay32.buffers)


def test_bucket_cut_lands_after_param():
    """[BUF] §4.3: cut when (param_end - bucket_start) >= bucket_size; the param is not split."""
    ps = [L.ParamSpec("a", 100), L.ParamSpec("b", 100), L.ParamSpec("c", 100)]
    lay = L.compute_layout(ps, L.LayoutConfig(bucket_size=150, dp_size=1, use_distributed_optimizer=False))
    # reverse order c, b, a: c ends at 100 (<150), b ends at 200 (>=150) -> cut; a alone
    assert [(b.offset, b.numel) for b in lay.buckets] == [(0, 200), (200, 100)]
    assert lay.param_index[1][2] == 0 and lay.param_index[0][2] == 1


def test_errors():
    with pytest.raises(ValueError):
        L.compute_layout([L.ParamSpec("z", 0)], L.LayoutConfig())
    with pytest.raises(ValueError):
        L.compute_layout([L.ParamSpec("a", 1)], L.LayoutConfig(dp_size=0))
    assert L.compute_layout([], L.LayoutConfig()).buffers == []
