"""The C++ layout engine (host-only, no GPU) is bit-exact with the oracle."""
import ctypes as C
import random

import pytest

from oracle import layout as L
from param_buffers_gb300 import abi, workloads as W
import param_buffers_gb300 as gtp

pytestmark = pytest.mark.skipif(not abi.LIB_PATH.exists(), reason="libgtp.so not built")


def both(params, cfg):
    ora = L.compute_layout([L.ParamSpec(f"p{i}", p.numel, p.dtype, p.quantized_storage, p.is_expert_parallel,
                                        p.is_layer_wise, p.is_shared_embedding) for i, p in enumerate(params)], cfg)
    nat = gtp.gtp_buffer_layout(params, gtp.LayoutConfig(cfg.bucket_size, cfg.dp_size, cfg.use_distributed_optimizer,
                                                         cfg.pad_buckets_for_high_nccl_busbw, cfg.grad_reduce_in_fp32))
    return ora, nat


def assert_same(ora, nat):
    assert len(ora.buffers) == len(nat.buffers)
    assert len(ora.buckets) == len(nat.buckets)
    for ob, nb in zip(ora.buffers, nat.buffers):
        assert ob.numel == nb["numel"]
        assert (ob.key.param_dtype, ob.key.grad_dtype) == (nb["param_dtype"], nb["grad_dtype"])
        assert (ob.key.is_expert_parallel, ob.key.is_layer_wise) == (bool(nb["is_expert_parallel"]), bool(nb["is_layer_wise"]))
        assert ob.buckets == list(range(nb["first_bucket"], nb["first_bucket"] + nb["num_buckets"]))
    for ok, nk in zip(ora.buckets, nat.buckets):
        assert (ok.offset, ok.numel_unpadded, ok.numel, ok.buffer_id, len(ok.params)) == \
            (nk["offset"], nk["numel_unpadded"], nk["numel"], nk["buffer_id"], nk["num_params"])
    for i, (s, e, b, buf) in ora.param_index.items():
        n = nat.index[i]
        bk = ora.buckets[b]
        assert (s, e, b, buf) == (n["start"], n["end"], n["bucket_id"], n["buffer_id"])
        assert bk.param_to_index[i] == (n["start_in_bucket"], n["end_in_bucket"])


def descs(params):
    return [gtp.ParamDesc(p.numel, p.dtype, is_shared_embedding=p.is_shared_embedding) for p in params]


@pytest.mark.parametrize("name", ["tiny", "layer", "stage", "7b", "7b_busbw", "7b_realistic", "toy"])
def test_workloads(name):
    if name == "toy":
        params, cfg = descs(W.toy_params()), L.LayoutConfig(bucket_size=None, dp_size=2, use_distributed_optimizer=False)
    elif name == "7b_realistic":
        params, cfg = descs(W.seven_b_realistic_params()), L.LayoutConfig(bucket_size=64_000_000, dp_size=64)
    else:
        bw = W.seven_b_buffer(True) if name == "7b_busbw" else W.BUFFERS[name]()
        params = descs(bw.params)
        cfg = L.LayoutConfig(bw.bucket_size, bw.dp_size, bw.use_distributed_optimizer, bw.pad_buckets_for_high_nccl_busbw)
    assert_same(*both(params, cfg))


@pytest.mark.parametrize("seed", range(300))
def test_random_lists(seed):
    rng = random.Random(1000 + seed)
    n = rng.randint(0, 40)
    params = [gtp.ParamDesc(rng.choice([1, 2, 7, 63, 64, 65, 127, 128, 1000, 4096, 100_003]),
                            rng.choice(["bf16", "bf16", "fp32", "fp16"]), quantized_storage=rng.random() < 0.1,
                            is_expert_parallel=rng.random() < 0.2, is_layer_wise=rng.random() < 0.1,
                            is_shared_embedding=rng.random() < 0.05) for _ in range(n)]
    cfg = L.LayoutConfig(bucket_size=rng.choice([None, 1, 100, 1000, 5000, 100_000]),
                         dp_size=rng.choice([1, 2, 3, 6, 8, 64, 96]),
                         use_distributed_optimizer=rng.random() < 0.7,
                         pad_buckets_for_high_nccl_busbw=rng.random() < 0.3,
                         grad_reduce_in_fp32=rng.random() < 0.7)
    assert_same(*both(params, cfg))


def test_capacity_protocol_and_errors():
    lib = abi.load()
    arr = (abi.gtp_param_desc * 3)(*[abi.gtp_param_desc(10, abi.GTP_BF16, 0, 0, 0, 0, 0) for _ in range(3)])
    cfg = abi.gtp_layout_config(15, 1, 0, 0, 1)
    nbuf, nbkt = C.c_int32(0), C.c_int32(0)
    assert lib.gtp_buffer_layout(arr, 3, C.byref(cfg), None, None, C.byref(nbuf), None, C.byref(nbkt)) == abi.GTP_OK
    assert (nbuf.value, nbkt.value) == (1, 2)
    bufs = (abi.gtp_buffer_desc * 1)()
    bkts = (abi.gtp_bucket_desc * 1)()
    nbuf2, nbkt2 = C.c_int32(1), C.c_int32(1)
    st = lib.gtp_buffer_layout(arr, 3, C.byref(cfg), None, bufs, C.byref(nbuf2), bkts, C.byref(nbkt2))
    assert st == abi.GTP_E_CAPACITY and nbkt2.value == 2
    assert b"capacity" in lib.gtp_last_error()
    def q(params, n, c):
        z1, z2 = C.c_int32(0), C.c_int32(0)
        return lib.gtp_buffer_layout(params, n, c, None, None, C.byref(z1), None, C.byref(z2))
    bad = (abi.gtp_param_desc * 1)(abi.gtp_param_desc(0, abi.GTP_BF16, 0, 0, 0, 0, 0))
    assert q(bad, 1, C.byref(cfg)) == abi.GTP_E_ARG
    bad = (abi.gtp_param_desc * 1)(abi.gtp_param_desc(5, 9, 0, 0, 0, 0, 0))
    assert q(bad, 1, C.byref(cfg)) == abi.GTP_E_DTYPE
    assert q(arr, 3, C.byref(abi.gtp_layout_config(15, 0, 0, 0, 1))) == abi.GTP_E_ARG
    assert q(arr, 3, None) == abi.GTP_E_ARG
    assert q(None, 2, C.byref(cfg)) == abi.GTP_E_ARG
    assert q(None, 0, C.byref(cfg)) == abi.GTP_OK
