"""Pins of the number-format oracle: two independent roundings agree, torch's casts agree
where they are defined, and hand-worked boundary cases."""
import numpy as np
import pytest
import torch

from oracle import floats as F


def adversarial_f32(n=200_000, seed=0):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
    specials = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.finfo(np.float32).max,
                         -np.finfo(np.float32).max, np.finfo(np.float32).tiny, 1e-45, -1e-45,
                         3.3895314e38, 65504.0, 448.0, 464.0, 2.0 ** -133, 2.0 ** -134], np.float32)
    # exact ties: bf16 value plus half an ulp (lower 16 bits = 0x8000), both parities
    ties = (rng.integers(0, 2 ** 16, size=4096, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    x = np.concatenate([bits.view(np.float32), specials, ties.view(np.float32)])
    return x[np.isfinite(x) | np.isinf(x)]


def test_bf16_integer_rounding_matches_torch():
    x = adversarial_f32()
    ours = F.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_two_roundings_agree():
    """Integer rounding of fp32 == grid rounding of the same value in float64."""
    x = adversarial_f32(seed=1)
    assert np.array_equal(F.f32_to_bf16_bits(x), F.f64_to_bf16_bits(x.astype(np.float64)))


def test_bf16_hand_cases():
    # 1 + 2^-8 is exactly half an ulp above 1.0 (even) -> 1.0; 1 + 3*2^-8 -> 1 + 2^-6 (even)
    assert F.f64_to_bf16_bits(1.0 + 2.0 ** -8) == 0x3F80
    assert F.f64_to_bf16_bits(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # just above the tie rounds up
    assert F.f64_to_bf16_bits(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    # largest finite bf16 and overflow to infinity
    assert F.f64_to_bf16_bits((2 - 2.0 ** -7) * 2.0 ** 127) == 0x7F7F
    assert F.f64_to_bf16_bits((2 - 2.0 ** -8) * 2.0 ** 127) == 0x7F80
    # smallest subnormal and the tie below it
    assert F.f64_to_bf16_bits(2.0 ** -133) == 0x0001
    assert F.f64_to_bf16_bits(2.0 ** -134) == 0x0000
    assert F.f64_to_bf16_bits(-2.0 ** -134) == 0x8000
    assert F.f32_to_bf16_bits(np.float32(np.nan)) & 0x7FC0 == 0x7FC0


def test_f64_to_bf16_single_rounding():
    """A value whose fp32 rounding would create a false tie rounds once, correctly."""
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40          # fp32(x) = 1 + 2^-8 (a tie) -> would give 1.0
    assert F.f64_to_bf16_bits(x) == 0x3F81
    assert F.f32_to_bf16_bits(np.float32(x)) == 0x3F80


def e4m3_table():
    codes = np.arange(256)
    vals = F.e4m3_decode(codes)
    return codes, vals


def test_e4m3_decode_definition():
    codes, vals = e4m3_table()
    assert vals[0x7E] == 448.0 and vals[0x08] == 2.0 ** -6 and vals[0x01] == 2.0 ** -9
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    assert vals[0x38] == 1.0 and vals[0xB8] == -1.0
    ref = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.nan_to_num(vals, nan=7.0), np.nan_to_num(ref, nan=7.0))


def test_e4m3_roundtrip_and_midpoints():
    codes, vals = e4m3_table()
    fin = ~np.isnan(vals)
    assert np.array_equal(F.e4m3_rne_satfinite(vals[fin]), codes[fin].astype(np.uint8))
    pos = np.sort(np.unique(vals[fin & (vals > 0)]))
    lo, hi = pos[:-1], pos[1:]
    mid = (lo + hi) / 2
    got = F.e4m3_decode(F.e4m3_rne_satfinite(mid))
    # ties go to the value with an even mantissa
    lo_codes = F.e4m3_rne_satfinite(lo)
    expect = np.where((lo_codes & 1) == 0, lo, hi)
    assert np.array_equal(got, expect)
    eps = (hi - lo) * 1e-6
    assert np.array_equal(F.e4m3_decode(F.e4m3_rne_satfinite(mid - eps)), lo)
    assert np.array_equal(F.e4m3_decode(F.e4m3_rne_satfinite(mid + eps)), hi)


def test_e4m3_matches_torch_inside_range():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100_000) * s for s in (1e-3, 0.05, 1, 30, 200)])
    x = x[np.abs(x) <= 448].astype(np.float32).astype(np.float64)
    ours = F.e4m3_rne_satfinite(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturation_and_specials():
    assert F.e4m3_rne_satfinite(449.0) == 0x7E
    assert F.e4m3_rne_satfinite(1e9) == 0x7E
    assert F.e4m3_rne_satfinite(-500.0) == 0xFE
    assert F.e4m3_rne_satfinite(np.nan) == 0x7F
    assert F.e4m3_rne_satfinite(-1e-5) == 0x80      # rounds to -0
    assert F.e4m3_rne_satfinite(2.0 ** -10) == 0x00  # tie between 0 and 2^-9 -> even (0)
    assert F.e4m3_rne_satfinite(3 * 2.0 ** -10) == 0x02


def test_e8m0():
    assert F.e8m0_value(127) == 1.0 and F.e8m0_value(0) == 2.0 ** -127 and F.e8m0_value(254) == 2.0 ** 127
    assert np.isnan(F.e8m0_value(255))
