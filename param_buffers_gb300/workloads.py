"""Seeded synthetic workloads: shapes, parameter lists and input generators.

This module holds no arithmetic of the method; it only describes the five workloads
and draws their inputs.  Both the CUDA path (bench, GPU tests) and the CPU oracle
(tests) take their inputs from here.

Workloads (the pages use mock data, "--mock-data", in the run.sh of the "Megatron-LM
architecture and source guide" page §4; no dataset is involved):

* ``tiny``   one column-parallel linear shard: W [512,256] ~N(0,0.02), X [128,256]
  ~N(0,1), dY [128,512] ~N(0,1), 2 microbatches; the flat buffer holds W and a
  512-element RMSNorm weight (ones).
* ``layer``  one Llama-3.2-1B layer at TP=2: QKV [1536,2048], O [2048,1024], fc1
  (gate+up) [8192,2048], fc2 [2048,4096]; seq 8192, micro-batch 1, 8 microbatches.
* ``stage``  the flat buffer of stage 0 of a TP=2/PP=2 split of the same model
  (embedding half plus 8 layers, 374,636,544 elements), 40M-element buckets, dp=2.
* ``7b``     a 1.875e9-element buffer: a tied embedding of 1,000,000 elements plus
  1,874 parameters of [1000,1000]; dp=64, bucket_size = max(40M, 64M).
* ``mxfp8``  FFN weights fp32 [8192,2048] and [2048,8192] ~N(0,0.02), X bf16
  [8192,2048] ~N(0,1).

Seeds: torch.Generator(seed = 1000 + workload index), tensors drawn in a fixed order.
Standard deviations are read as standard deviations (N(0, 1e-3) has std 1e-3).
"""
from __future__ import annotations

from dataclasses import dataclass, field

WORKLOADS = ("tiny", "layer", "stage", "7b", "mxfp8")
SEED_BASE = 1000


def seed_of(name: str) -> int:
    return SEED_BASE + WORKLOADS.index(name)


# --------------------------------------------------------------------------- linear GEMMs

@dataclass(frozen=True)
class LinearShape:
    name: str
    N: int   # out-features of the TP shard (rows of W)
    K: int   # in-features of the TP shard


TINY_LINEAR = LinearShape("W", 512, 256)
TINY_M = 128
TINY_MICROBATCHES = 2

LAYER_LINEARS = (
    LinearShape("qkv", 1536, 2048),
    LinearShape("proj", 2048, 1024),
    LinearShape("fc1", 8192, 2048),
    LinearShape("fc2", 2048, 4096),
)
LAYER_M = 8192          # seq 8192 x micro-batch 1
LAYER_MICROBATCHES = 8
HIDDEN = 2048


def linear_flops(M: int, N: int, K: int) -> int:
    """2*M*N*K for one of the three GEMMs."""
    return 2 * M * N * K


# --------------------------------------------------------------------------- buffers

@dataclass(frozen=True)
class Param:
    name: str
    numel: int
    dtype: str = "bf16"
    is_shared_embedding: bool = False


@dataclass(frozen=True)
class BufferWorkload:
    name: str
    params: tuple            # model order
    bucket_size: int | None
    dp_size: int
    use_distributed_optimizer: bool = True
    pad_buckets_for_high_nccl_busbw: bool = False
    gradient_scaling_factor: float = 1.0
    grad_std: float = 1e-3
    param_std: float = 0.02
    hparams: dict = field(default_factory=lambda: dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8,
                                                       weight_decay=0.1))


def _layer_params(prefix: str) -> list:
    return [Param(f"{prefix}input_norm", HIDDEN), Param(f"{prefix}qkv", 1536 * 2048),
            Param(f"{prefix}proj", 2048 * 1024), Param(f"{prefix}mlp_norm", HIDDEN),
            Param(f"{prefix}fc1", 8192 * 2048), Param(f"{prefix}fc2", 2048 * 4096)]


def tiny_buffer() -> BufferWorkload:
    return BufferWorkload("tiny", (Param("W", 512 * 256), Param("norm", 512)), bucket_size=40_000_000,
                          dp_size=2, gradient_scaling_factor=0.5)


def layer_buffer() -> BufferWorkload:
    return BufferWorkload("layer", tuple(_layer_params("")), bucket_size=40_000_000, dp_size=2,
                          gradient_scaling_factor=0.5)


def stage_buffer() -> BufferWorkload:
    ps = [Param("embedding", 64128 * 2048)]
    for i in range(8):
        ps += _layer_params(f"layers.{i}.")
    return BufferWorkload("stage", tuple(ps), bucket_size=40_000_000, dp_size=2, gradient_scaling_factor=0.5)


def seven_b_buffer(busbw: bool = False) -> BufferWorkload:
    ps = [Param("embedding", 1_000_000, is_shared_embedding=True)]
    ps += [Param(f"w{i}", 1_000_000) for i in range(1874)]
    return BufferWorkload("7b", tuple(ps), bucket_size=max(40_000_000, 1_000_000 * 64), dp_size=64,
                          pad_buckets_for_high_nccl_busbw=busbw, gradient_scaling_factor=1.0 / 64)


def seven_b_realistic_params() -> tuple:
    """Layout-only list: tied embedding half [64128,2048] plus 57 TP=2 Llama layers."""
    ps = [Param("embedding", 64128 * 2048, is_shared_embedding=True)]
    for i in range(57):
        ps += _layer_params(f"layers.{i}.")
    return tuple(ps)


def toy_params() -> tuple:
    """The 2-rank toy buffer of the guide's §6.3: W1 (6), W2 (4), WL (12) in model order."""
    return (Param("W1", 6), Param("W2", 4), Param("WL", 12))


BUFFERS = {"tiny": tiny_buffer, "layer": layer_buffer, "stage": stage_buffer, "7b": seven_b_buffer}

MXFP8_W = (("fc1", 8192, 2048), ("fc2", 2048, 8192))
MXFP8_X = (8192, 2048)


# --------------------------------------------------------------------------- generators

def generator(seed: int, device="cpu"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, std: float, g, device="cpu"):
    """N(0, std) drawn in fp32 and stored as bf16 (torch's own fp32 -> bf16 cast)."""
    import torch
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def randn_f32(shape, std: float, g, device="cpu"):
    import torch
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def linear_inputs(M: int, N: int, K: int, g, device="cpu", w_std: float = 0.02):
    """(X [M,K], W [N,K], dY [M,N]) in bf16, drawn in that order."""
    X = randn_bf16((M, K), 1.0, g, device)
    W = randn_bf16((N, K), w_std, g, device)
    dY = randn_bf16((M, N), 1.0, g, device)
    return X, W, dY


def buffer_state(numel: int, g, device="cpu", grad_std: float = 1e-3, param_std: float = 0.02):
    """Step-1 state of a flat buffer: grad fp32 ~N(0, grad_std); bf16 params ~N(0, param_std);
    fp32 master = float(param); m = v = 0.  Returns (grad, master, m, v, param)."""
    import torch
    grad = randn_f32((numel,), grad_std, g, device)
    param = randn_bf16((numel,), param_std, g, device)
    master = param.float()
    m = torch.zeros(numel, dtype=torch.float32, device=device)
    v = torch.zeros(numel, dtype=torch.float32, device=device)
    return grad, master, m, v, param
