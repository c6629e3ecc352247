"""Gradient norm, non-finite check and clip coefficient (oracle; test infrastructure).

[BUF] §6.3: with check_for_nan_in_grad / check_for_large_grads, start_grad_sync computes
each bucket's gradient L2 norm before the collective; NaN/Inf is fatal, an abnormally large
norm non-fatal.  [MLM] §4 trains with --clip-grad 1.0 and optimizer.step() returns
grad_norm.

Reading (R13): the norm is taken of the scaled gradient v = factor_b * g of each bucket
(what the optimizer consumes); the global norm is sqrt(sum_b ||v_b||^2) and clipping
multiplies every gradient by coef = min(1, max_norm / (norm + 1e-6)) (1 when max_norm is
0), the usual global-norm rule.  The optimizer applies it after the bucket scale.
"""
from __future__ import annotations

import math

import numpy as np


def bucket_sumsq(grad_f32: np.ndarray, buckets, factors) -> np.ndarray:
    """||factor_b * g||^2 per bucket, the products and their squares exact in float64.

    ``buckets`` is a sequence of (offset, numel); factors are the fp32 values the kernel
    receives.
    """
    out = np.zeros(len(buckets), np.float64)
    for i, ((off, n), f) in enumerate(zip(buckets, factors)):
        v = grad_f32[off:off + n].astype(np.float64) * np.float64(np.float32(f))
        out[i] = float(np.dot(v, v))
    return out


def bucket_nonfinite(grad_f32: np.ndarray, buckets, factors) -> np.ndarray:
    out = np.zeros(len(buckets), np.int64)
    for i, ((off, n), f) in enumerate(zip(buckets, factors)):
        v = grad_f32[off:off + n].astype(np.float64) * np.float64(np.float32(f))
        out[i] = int(np.count_nonzero(~np.isfinite(v)))
    return out


def total_norm(sumsq) -> float:
    return math.sqrt(float(np.sum(sumsq)))


def clip_coef(norm: float, max_norm: float) -> float:
    """min(1, max_norm / (norm + 1e-6)); clipping off when max_norm == 0."""
    if max_norm <= 0:
        return 1.0
    return min(1.0, max_norm / (norm + 1e-6))
