"""Flat param/grad buffer layout (oracle; test infrastructure).

Follows [BUF] §3 (BufferKey grouping), §4.1 (reverse order), §4.2 (alignment and
padding), §4.3 (bucket_size and the cut rule) and §5 (param_index_map, bucket views),
and [MLM] §6.3 (the same construction, with the 2-rank toy buffer).

Rules, in the pages' terms:

1. Every ``requires_grad`` parameter is grouped by
   BufferKey(param_dtype, grad_dtype, is_expert_parallel, is_layer_wise); one physical
   buffer per distinct key, keys in order of first appearance ([BUF] §3).
   param_dtype is the storage dtype (FP8 / NVFP4 params key as uint8); grad_dtype is
   fp32 when grad_reduce_in_fp32 else the parameter's dtype.
2. Parameters are placed in reverse model order (backprop order), so offset 0 holds
   the tail of the model ([BUF] §4.1).
3. Without the distributed optimizer there is no padding at all: a parameter starts
   where the previous one ended, numel == numel_unpadded ([BUF] §4.2).
4. With the distributed optimizer each parameter start is rounded up to a multiple of
   64 *elements* (the page corrects a docstring that says bytes), and each bucket end
   is rounded up to lcm(dp, 128), or lcm(dp, 128, 2**16) with
   pad_buckets_for_high_nccl_busbw, so every bucket divides evenly by dp ([BUF] §4.2).
5. A bucket is closed right after the parameter whose end reaches
   ``end - bucket_start >= bucket_size`` ([BUF] §4.3); bucket_size is in elements.
   ``None`` means one bucket.
6. With the distributed optimizer a ``shared_embedding`` parameter closes any open
   bucket, occupies a new bucket alone, and closes it ([BUF] §4.2).

Readings where the pages leave a step open (each is listed in the design notes):

* R3: the cut test uses the unpadded parameter end; default mode has no start
  padding (the toy forces this: W2 starts at 12, not 64).
* R3b: a parameter never straddles two buckets.  [BUF] §4.3 says a parameter "can
  span two buckets", but the cut lands after the parameter by rule 5, and
  param_index_map carries a single bucket id per parameter (§5); the sentence is read
  as the dp *shards*, which do cut parameters.
* R11: the shared-embedding isolation of rule 6 is applied in distributed-optimizer
  mode only; the page lists it among the dist-opt layout rules (§4.2 table), whose
  motivation is equal shards on the two pipeline stages.

Parity unpinned: the toy's "param_data sum=-4.6088" ([MLM] §6.4) needs seeds and
values the page does not give.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

DTYPES = ("fp32", "bf16", "fp16", "uint8")


@dataclass(frozen=True)
class ParamSpec:
    name: str
    numel: int
    dtype: str = "bf16"              # logical dtype of the parameter
    quantized_storage: bool = False  # FP8 / NVFP4 parameter: stored as uint8
    is_expert_parallel: bool = False
    is_layer_wise: bool = False
    is_shared_embedding: bool = False


@dataclass(frozen=True)
class LayoutConfig:
    bucket_size: Optional[int] = None       # elements; None = a single bucket
    dp_size: int = 1
    use_distributed_optimizer: bool = True
    pad_buckets_for_high_nccl_busbw: bool = False
    grad_reduce_in_fp32: bool = True


@dataclass(frozen=True)
class BufferKey:
    param_dtype: str
    grad_dtype: str
    is_expert_parallel: bool
    is_layer_wise: bool


@dataclass
class Bucket:
    buffer_id: int
    offset: int
    numel_unpadded: int
    numel: int
    params: list = field(default_factory=list)          # param indices (model list)
    param_to_index: dict = field(default_factory=dict)  # param idx -> (start, end) within bucket


@dataclass
class Buffer:
    key: BufferKey
    numel: int
    params: list                      # param indices in model order
    buckets: list                     # global bucket indices


@dataclass
class Layout:
    buffers: list
    buckets: list
    param_index: dict                 # param idx -> (start, end, bucket_id, buffer_id)


def default_bucket_size(dp_size: int) -> int:
    """max(40M, 1M * dp) elements ([BUF] §4.3)."""
    return max(40_000_000, 1_000_000 * dp_size)


def bucket_size_for_num_buckets(num_parameters: int, num_buckets: int) -> int:
    """The num_buckets variant: bucket_size = num_parameters // num_buckets ([BUF] §4.3)."""
    return num_parameters // num_buckets


def buffer_key(p: ParamSpec, cfg: LayoutConfig) -> BufferKey:
    """[BUF] §3: the four dimensions of BufferKey."""
    param_dtype = "uint8" if p.quantized_storage else p.dtype
    grad_dtype = "fp32" if cfg.grad_reduce_in_fp32 else p.dtype
    return BufferKey(param_dtype, grad_dtype, p.is_expert_parallel, p.is_layer_wise)


def group_params_for_buffers(params: Sequence[ParamSpec], cfg: LayoutConfig) -> dict:
    groups: dict = {}
    for i, p in enumerate(params):
        groups.setdefault(buffer_key(p, cfg), []).append(i)
    return groups


def round_up(x: int, d: int) -> int:
    return -(-x // d) * d


def bucket_end_divisor(cfg: LayoutConfig) -> int:
    """lcm(dp, 128), or lcm(dp, 128, 2**16) with the busbw option ([BUF] §4.2)."""
    d = math.lcm(cfg.dp_size, 128)
    if cfg.pad_buckets_for_high_nccl_busbw:
        d = math.lcm(d, 2 ** 16)
    return d


def compute_layout(params: Sequence[ParamSpec], cfg: LayoutConfig) -> Layout:
    if cfg.dp_size < 1:
        raise ValueError("dp_size must be >= 1")
    if cfg.bucket_size is not None and cfg.bucket_size <= 0:
        raise ValueError("bucket_size must be positive or None")
    for p in params:
        if p.numel <= 0:
            raise ValueError(f"parameter {p.name} has no elements")
        if p.dtype not in DTYPES:
            raise ValueError(f"unknown dtype {p.dtype}")

    distopt = cfg.use_distributed_optimizer
    divisor = bucket_end_divisor(cfg) if distopt else 1

    buffers: list[Buffer] = []
    buckets: list[Bucket] = []
    index: dict = {}

    for key, members in group_params_for_buffers(params, cfg).items():
        buffer_id = len(buffers)
        buf = Buffer(key=key, numel=0, params=list(members), buckets=[])
        buffers.append(buf)

        bucket_start = 0        # offset of the open bucket
        cur = 0                 # first free element
        open_params: list = []

        def close(end_unpadded: int) -> int:
            nonlocal bucket_start, open_params
            end = round_up(end_unpadded, divisor) if distopt else end_unpadded
            b = Bucket(buffer_id=buffer_id, offset=bucket_start,
                       numel_unpadded=end_unpadded - bucket_start,
                       numel=end - bucket_start, params=list(open_params))
            bid = len(buckets)
            for pi in open_params:
                s, e = index[pi][0], index[pi][1]
                index[pi] = (s, e, bid, buffer_id)
                b.param_to_index[pi] = (s - bucket_start, e - bucket_start)
            buckets.append(b)
            buf.buckets.append(bid)
            bucket_start = end
            open_params = []
            return end

        for pi in reversed(members):                    # backprop order ([BUF] §4.1)
            p = params[pi]
            isolate = distopt and p.is_shared_embedding
            if isolate and open_params:
                cur = close(cur)
            start = round_up(cur, 64) if distopt else cur
            end = start + p.numel
            index[pi] = (start, end, -1, buffer_id)
            open_params.append(pi)
            cur = end
            if isolate or (cfg.bucket_size is not None and end - bucket_start >= cfg.bucket_size):
                cur = close(end)
        if open_params:
            cur = close(cur)
        buf.numel = cur
    return Layout(buffers=buffers, buckets=buckets, param_index=index)


def shard_param_ranges(layout: Layout, buffer_id: int, dp_size: int, dp_rank: int) -> list[dict]:
    """The range map of one dp rank ([BUF] §6.5, [MLM] §6.4): for every parameter that overlaps
    the rank's shard of its bucket, the overlap as buffer ("world"), in-bucket, shard-local and
    in-parameter offsets.  Ordered by bucket, then position."""
    out = []
    for bid in layout.buffers[buffer_id].buckets:
        b = layout.buckets[bid]
        s0, s1 = shard_ranges(b, dp_size)[dp_rank]
        for pi in sorted(b.params, key=lambda i: layout.param_index[i][0]):
            ps, pe = layout.param_index[pi][:2]
            lo, hi = max(ps, s0), min(pe, s1)
            if lo < hi:
                out.append({"param": pi, "bucket_id": bid, "world_start": lo, "world_end": hi,
                            "bucket_start": lo - b.offset, "local_start": lo - s0, "param_start": lo - ps})
    return out


def shard_ranges(bucket: Bucket, dp_size: int) -> list[tuple[int, int]]:
    """The dp equal element shards of one bucket, rank r owning the r-th ([BUF] §6.5).

    The shards ignore parameter boundaries ([BUF] §4.3, [MLM] §6.4).
    """
    if bucket.numel % dp_size:
        raise ValueError("bucket numel is not divisible by dp")
    n = bucket.numel // dp_size
    return [(bucket.offset + r * n, bucket.offset + (r + 1) * n) for r in range(dp_size)]
