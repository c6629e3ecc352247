"""The optimizer half of the step over the flat buffer (oracle; test infrastructure).

Steps, in the order the pages give them:

* zero: ``zero_grad_buffer()`` zeroes all of ``grad_data`` at the start of each
  iteration, without freeing it ([BUF] §6.6, §8).
* scale: ``start_grad_sync`` first multiplies each bucket's ``grad_data`` by its
  ``gradient_scaling_factor`` (1/dp by default) ([BUF] §6.3, §3).
* grad -> fp32: ``shard_main_param.grad = shard_model_grad.float()`` ([BUF] §6.5 ①,
  [MLM] §6.4 step 1) - the identity for an fp32 grad buffer.
* Adam on the fp32 master and m, v ([BUF] §6.5 ②, [MLM] §6.4 step 2), with the
  run.sh hyper-parameters lr 3e-4, beta1 0.9, beta2 0.95, weight decay 0.1
  ([MLM] §4).
* cast: the updated fp32 master is copied into ``param_data`` as bf16
  ([BUF] §6.5 ③, [MLM] §6.4 step 3).

Reading R4: the Adam variant is AdamW, i.e. decoupled weight decay with bias
correction (wd = 0 gives Adam); no decay exclusion for 1-D parameters (the pages
only give ``--weight-decay 0.1``).  eps = 1e-8.
Reading R9: padding elements go through the same update; with zero grad, master, m
and v they stay exactly zero.
Reading R10: the fused sweep orders the steps scale -> Adam -> cast -> zero the
grad; zeroing right after the step is equivalent to zeroing at the start of the
next iteration.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from .floats import f32_to_bf16_bits


@dataclass(frozen=True)
class AdamWHparams:
    lr: float = 3e-4
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1


def adamw_element(p: float, g: float, m: float, v: float, t: int, h: AdamWHparams):
    """One AdamW update of one element, float64, written out term by term.

    m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2
    m_hat = m / (1 - b1^t);  v_hat = v / (1 - b2^t)
    p <- p (1 - lr wd) - lr m_hat / (sqrt(v_hat) + eps)
    """
    m = h.beta1 * m + (1.0 - h.beta1) * g
    v = h.beta2 * v + (1.0 - h.beta2) * g * g
    m_hat = m / (1.0 - h.beta1 ** t)
    v_hat = v / (1.0 - h.beta2 ** t)
    p = p * (1.0 - h.lr * h.weight_decay) - h.lr * m_hat / (math.sqrt(v_hat) + h.eps)
    return p, m, v


def adamw(p, g, m, v, t: int, h: AdamWHparams):
    """The same update on arrays (float64 in, float64 out)."""
    p = np.asarray(p, np.float64)
    g = np.asarray(g, np.float64)
    m = np.asarray(m, np.float64)
    v = np.asarray(v, np.float64)
    m = h.beta1 * m + (1.0 - h.beta1) * g
    v = h.beta2 * v + (1.0 - h.beta2) * g * g
    m_hat = m / (1.0 - h.beta1 ** t)
    v_hat = v / (1.0 - h.beta2 ** t)
    p = p * (1.0 - h.lr * h.weight_decay) - h.lr * m_hat / (np.sqrt(v_hat) + h.eps)
    return p, m, v


def adamw_loop(p, g, m, v, t: int, h: AdamWHparams):
    """``adamw_element`` over every element (small inputs; the literal scalar form)."""
    P = np.empty(len(p)); Mo = np.empty(len(p)); Vo = np.empty(len(p))
    for i in range(len(p)):
        P[i], Mo[i], Vo[i] = adamw_element(float(p[i]), float(g[i]), float(m[i]), float(v[i]), t, h)
    return P, Mo, Vo


def bucket_factor_per_element(numel: int, buckets, factors) -> np.ndarray:
    """The gradient_scaling_factor that applies to each element of grad_data.

    ``buckets`` is a sequence of (offset, numel) ranges; elements outside every bucket
    (none, for a layout's own bucket list) keep factor 1.
    """
    f = np.ones(numel, np.float64)
    for (off, n), fac in zip(buckets, factors):
        f[off:off + n] = fac
    return f


def scale_grad(grad_f32: np.ndarray, factor: np.ndarray) -> np.ndarray:
    """grad_data *= factor, rounded to fp32 as an in-place fp32 multiply is."""
    return (grad_f32.astype(np.float64) * factor).astype(np.float32)


def fused_sweep(grad, master, exp_avg, exp_avg_sq, factor, t: int, h: AdamWHparams):
    """scale -> (.float()) -> AdamW -> bf16 cast -> zero grad, per element.

    Returns (grad_out, master64, m64, v64, param_bf16_of_master64_rounded_to_fp32).
    The master / m / v results are float64 (the exact update of the fp32 inputs); the
    bf16 param is the RNE cast of the fp32-rounded master, as the path stores it.
    """
    g = scale_grad(grad, factor).astype(np.float64)
    p, m, v = adamw(master, g, exp_avg, exp_avg_sq, t, h)
    param = f32_to_bf16_bits(p.astype(np.float32))
    return np.zeros_like(grad), p, m, v, param


def fused_sweep_mxfp8(grad, master, exp_avg, exp_avg_sq, factor, t: int, h: AdamWHparams):
    """The sweep of a native-MXFP8 parameter buffer ([GTP] §1.3: the optimizer writes the
    FP8 weight from the fp32 master once per step): as ``fused_sweep``, but param_data
    holds the MX blocks (E4M3 codes, E8M0 scales) of the fp32-rounded master instead of
    its bf16 cast.  Returns (grad_out, master64, m64, v64, codes, scales)."""
    from .mxfp8 import quantize_flat_blocks
    g = scale_grad(grad, factor).astype(np.float64)
    p, m, v = adamw(master, g, exp_avg, exp_avg_sq, t, h)
    codes, scales = quantize_flat_blocks(p.astype(np.float32))
    return np.zeros_like(grad), p, m, v, codes, scales
