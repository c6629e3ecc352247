"""Pins of oracle/rs_sum.py (the local fp32 sum of the all-to-all reduce-scatter, [BUF] §9.1)
against closed forms, library special cases and hand-worked roundings."""
import numpy as np
import torch

from oracle import floats as F
from oracle import rs_sum as R


def test_small_integers_sum_exactly():
    """Integers below 2^24 add exactly in fp32: the sum is the integer sum, any order."""
    rng = np.random.default_rng(0)
    slices = [rng.integers(-1000, 1000, 4096).astype(np.float32) for _ in range(64)]
    exact = np.sum(np.stack(slices).astype(np.int64), axis=0)
    assert np.array_equal(R.local_sum_fp32(slices), exact.astype(np.float32))


def test_one_rounding_per_addition_in_rank_order():
    """2^24 + 1 rounds to 2^24 (a tie, to even): in rank order [2^24, 1, 1] the sum stays
    2^24, while [1, 1, 2^24] reaches 2^24 + 2 exactly -- the order and the per-addition
    rounding of the reading, worked by hand."""
    big = np.float32(2.0 ** 24)
    a = R.local_sum_fp32([np.array([big]), np.array([np.float32(1)]), np.array([np.float32(1)])])
    b = R.local_sum_fp32([np.array([np.float32(1)]), np.array([np.float32(1)]), np.array([big])])
    assert a[0] == np.float32(2.0 ** 24)
    assert b[0] == np.float32(2.0 ** 24 + 2)


def test_error_within_the_recursive_summation_bound_and_not_exact():
    """Against the exact (float64) sum of bf16 slices: inside the (P-1) 2^-24 sum|x| bound,
    and not equal to it everywhere (fp32, not a wider accumulator)."""
    rng = np.random.default_rng(1)
    slices = [F.f32_to_bf16_bits((rng.standard_normal(20000) * np.exp2(rng.integers(-20, 20, 20000)))
                                 .astype(np.float32)) for _ in range(64)]
    got = R.local_sum_fp32(slices).astype(np.float64)
    exact = np.sum([F.bf16_bits_to_f64(s) for s in slices], axis=0)
    assert np.all(np.abs(got - exact) <= R.sum_bound(slices))
    assert np.any(got != exact)


def test_bf16_output_is_the_rne_cast_of_the_fp32_sum():
    """The bf16 output equals torch's float32 -> bfloat16 cast (round to nearest even) of
    the fp32 sum."""
    rng = np.random.default_rng(2)
    slices = [F.f32_to_bf16_bits(rng.standard_normal(8192).astype(np.float32)) for _ in range(8)]
    f32 = R.local_sum_fp32(slices)
    want = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(R.local_sum(slices, out_bf16=True), want)
    assert np.array_equal(R.local_sum(slices, out_bf16=False), f32)


def test_one_slice_is_the_cast_and_specials_propagate():
    x = F.f32_to_bf16_bits(np.array([1.5, -0.0, np.inf, 3e38], np.float32))
    assert np.array_equal(R.local_sum([x], out_bf16=True), x)
    nan = np.array([np.nan, np.inf, 1.0], np.float32)
    other = np.array([1.0, -np.inf, np.float32(3.4e38)], np.float32)
    out = R.local_sum_fp32([nan, other, other])
    assert np.isnan(out[0]) and np.isnan(out[1])       # NaN stays NaN; +inf + -inf is NaN
    assert np.isinf(out[2]) and out[2] > 0              # overflow to +inf in fp32
