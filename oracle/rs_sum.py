"""The local fp32 sum of the all-to-all reduce-scatter (oracle; test infrastructure).

[BUF] §9.1 (reduce_scatter_with_fp32_accumulation): the bucket's reduce-scatter becomes an
all-to-all -- every rank sends each dp rank that rank's slice of its low-precision grad
bucket -- and, when the exchange completes, each rank adds up the world_size slices it
received with an fp32 sum and casts the result back to the output's dtype.

Reading R20: the fp32 sum adds the slices in rank order, one fp32 rounding per addition
(a sequential fp32 accumulation that starts from slice 0 converted exactly to fp32); the
pages name the sum's precision, not its order.  The total is then rounded once to the
output dtype (round-to-nearest-even to bf16, or kept as fp32).

Slices are given as bf16 bit patterns (uint16) or float32 arrays of equal length.
"""
from __future__ import annotations

import numpy as np

from .floats import bf16_bits_to_f32, f32_to_bf16_bits


def _as_f32(s: np.ndarray) -> np.ndarray:
    s = np.asarray(s)
    if s.dtype == np.uint16:
        return bf16_bits_to_f32(s)              # bf16 -> fp32 is exact
    return s.astype(np.float32)


def local_sum_fp32(slices) -> np.ndarray:
    """sum_r slices[r] in fp32, r = 0, 1, ..., P-1, rounded after every addition."""
    acc = _as_f32(slices[0]).copy()
    with np.errstate(over="ignore", invalid="ignore"):   # inf and NaN are values here, not errors
        for s in slices[1:]:
            acc = (acc + _as_f32(s)).astype(np.float32)   # one IEEE fp32 addition, round to nearest even
    return acc


def local_sum(slices, out_bf16: bool) -> np.ndarray:
    """The rank's reduced shard: the fp32 sum cast to the output dtype (bf16 bit patterns or
    float32)."""
    acc = local_sum_fp32(slices)
    return f32_to_bf16_bits(acc) if out_bf16 else acc


def sum_bound(slices) -> np.ndarray:
    """|fp32 sequential sum - exact sum| <= (P - 1) 2^-24 sum_r |x_r| per element (each of the
    P - 1 additions rounds by at most half an ulp of a partial sum no larger than the sum of
    magnitudes; the textbook bound of recursive summation)."""
    mags = np.sum([np.abs(_as_f32(s).astype(np.float64)) for s in slices], axis=0)
    return (len(slices) - 1) * 2.0 ** -24 * mags
