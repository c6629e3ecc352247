"""Parameter counts of the Llama-3.2-1B shape (oracle; test infrastructure).

[MLM] §1 (overview) states the shape: L=16 layers, h=2048, f=8192, 32 query heads,
8 K/V heads, head width 64, vocabulary 128256, untied input embedding and output
layer.  Per layer the Q,K,V,O weights hold 2h**2 + 2h(n_kv d_h) parameters, the
SwiGLU gate/up/down weights 3hf, and the two RMSNorm weights 2h.

Reading (listed as R1): the page's total of about 1,498,482,688 exceeds
16 * layer + 2 * v * h by exactly 2,048 = h; that is taken to be the final RMSNorm.

Reading (listed as R8): the order of parameters inside a layer is the pre-norm
execution order input_norm, qkv, proj, mlp_norm, fc1 (gate+up), fc2 (down); the
pages do not give ``named_parameters`` order.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class LlamaShape:
    num_layers: int = 16
    hidden: int = 2048
    ffn: int = 8192
    n_q: int = 32
    n_kv: int = 8
    d_head: int = 64
    vocab: int = 128256
    tied: bool = False
    final_norm: bool = True


LLAMA_32_1B = LlamaShape()


def layer_params(s: LlamaShape) -> int:
    """2h^2 + 2h(n_kv d_h) + 3hf + 2h ([MLM] §1)."""
    h = s.hidden
    return 2 * h * h + 2 * h * (s.n_kv * s.d_head) + 3 * h * s.ffn + 2 * h


def embedding_params(s: LlamaShape) -> int:
    """v*h for the input embedding, and again for the untied output layer ([MLM] §1)."""
    return s.vocab * s.hidden


def total_params(s: LlamaShape) -> int:
    n = s.num_layers * layer_params(s) + embedding_params(s) * (1 if s.tied else 2)
    if s.final_norm:
        n += s.hidden
    return n


def tp_layer_tensors(s: LlamaShape, tp: int) -> list[tuple[str, tuple[int, ...]]]:
    """The tensors one TP rank holds for one layer, in the order of reading R8.

    Column-parallel weights are split on the output dimension, [out/TP, in]; row-parallel
    weights on the input dimension, [out, in/TP] ([LIN] §1, [MLM] §6.2).  The QKV and
    gate+up projections are column-parallel, proj and down are row-parallel; RMSNorm
    weights are replicated across the TP group.
    """
    h, f = s.hidden, s.ffn
    qkv_out = (s.n_q + 2 * s.n_kv) * s.d_head
    return [
        ("input_norm", (h,)),
        ("qkv", (qkv_out // tp, h)),
        ("proj", (h, s.n_q * s.d_head // tp)),
        ("mlp_norm", (h,)),
        ("fc1", (2 * f // tp, h)),
        ("fc2", (h, f // tp)),
    ]


def tp_pp_stage0_tensors(s: LlamaShape, tp: int, pp: int) -> list[tuple[str, tuple[int, ...]]]:
    """Stage 0 of a TP x PP split: the vocab-parallel input embedding half plus L/PP layers."""
    out = [("embedding", (s.vocab // tp, s.hidden))]
    for i in range(s.num_layers // pp):
        out += [(f"layers.{i}.{n}", shp) for n, shp in tp_layer_tensors(s, tp)]
    return out


def numel(shape: tuple[int, ...]) -> int:
    n = 1
    for d in shape:
        n *= d
    return n
