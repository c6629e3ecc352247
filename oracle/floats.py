"""Number formats used on the path, written from their definitions (oracle; test infrastructure).

* bf16: 1 sign, 8 exponent (bias 127), 7 stored mantissa bits.  The casts in
  [MLM] §6.4 step 3 ("fp32 master shard -> param_data, cast to bf16") and
  [BUF] §6.5 step ③ write bf16 params from fp32 masters; the rounding is
  round-to-nearest, ties-to-even (RNE), the IEEE default, since the pages name no other.
* E4M3 (OCP FP8, "fn" flavour): 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
  infinities, NaN = S.1111.111, largest finite 1.75 * 2**8 = 448, smallest
  subnormal 2**-9.  Used for the MXFP8 weights of [GTP] §1.3.
* E8M0: an unsigned biased power-of-two exponent, value 2**(byte - 127), 0xFF = NaN.
  One per 32-element block ([GTP] §1.3, table "Communication volume breakdown":
  block 32, scale 1/32 byte per element).
* E2M1 (FP4): 1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes 0, 0.5, 1, 1.5,
  2, 3, 4, 6; no infinity or NaN.  The NVFP4 elements of [GTP] §1.3 ("packed 4-bit,
  kFloat4E2M1").

Two independent ways of rounding are written here so that tests can check them
against each other: integer bit manipulation on the fp32 encoding, and exact
power-of-two scaling in float64 followed by round-half-even to an integer grid.
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------- bf16

def f32_bits(x) -> np.ndarray:
    """The uint32 encoding of float32 values."""
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)


def bf16_bits_to_f32(b) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    b = np.asarray(b).astype(np.uint32)
    return (b << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(b) -> np.ndarray:
    return bf16_bits_to_f32(b).astype(np.float64)


def f32_to_bf16_bits(x) -> np.ndarray:
    """RNE float32 -> bf16 by integer arithmetic on the fp32 encoding.

    The upper 16 bits are kept; the lower 16 decide the rounding: above half an ulp
    rounds up, below rounds down, exactly half rounds to the even upper half.  A carry
    out of the mantissa moves into the exponent, which is the correct result (up to
    and including overflow to infinity).  NaNs keep their sign and become quiet NaNs.
    """
    u = f32_bits(x).astype(np.uint64)
    upper = u >> np.uint64(16)
    lower = u & np.uint64(0xFFFF)
    half = np.uint64(0x8000)
    up = (lower > half) | ((lower == half) & ((upper & np.uint64(1)) == np.uint64(1)))
    out = upper + up.astype(np.uint64)
    is_nan = ((u & np.uint64(0x7F800000)) == np.uint64(0x7F800000)) & ((u & np.uint64(0x7FFFFF)) != 0)
    out = np.where(is_nan, upper | np.uint64(0x0040), out)
    return out.astype(np.uint16)


def _round_to_grid_rne(x: np.ndarray, frac_bits: int, min_exp: int) -> np.ndarray:
    """Round float64 values to a binary floating-point grid, ties to even.

    The grid has ``frac_bits`` stored fraction bits and smallest normal exponent
    ``min_exp`` (below which the spacing stays 2**(min_exp - frac_bits): subnormals).
    For each x the spacing of the grid around |x| is a power of two, so x / spacing is
    exact in float64 and ``np.rint`` (round half to even) does the rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    with np.errstate(divide="ignore", invalid="ignore"):
        _, e = np.frexp(ax)                 # ax = m * 2**e, m in [0.5, 1)
    exp = np.maximum(e - 1, min_exp)        # floor(log2 ax), clamped into the subnormal range
    spacing_exp = exp - frac_bits
    q = np.ldexp(ax, -spacing_exp)          # exact: scaling by a power of two
    r = np.ldexp(np.rint(q), spacing_exp)
    return np.copysign(r, x)


def f64_to_bf16_bits(x) -> np.ndarray:
    """RNE float64 -> bf16 in one rounding (no intermediate float32 rounding)."""
    x = np.asarray(x, dtype=np.float64)
    r = _round_to_grid_rne(np.where(np.isfinite(x), x, 0.0), frac_bits=7, min_exp=-126)
    with np.errstate(over="ignore"):
        # bf16's largest finite value is (2 - 2**-7) * 2**127; a rounded magnitude of
        # 2**128 or more is infinity.
        r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, r), r)
        r = np.where(np.isfinite(x), r, x)
        r32 = r.astype(np.float32)          # exact: r lies on the bf16 grid (or is inf/nan)
    bits = (f32_bits(r32) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    return np.where(nan, (bits | np.uint16(0x0040)), bits).astype(np.uint16)


# ----------------------------------------------------------------------------- E4M3

E4M3_MAX = 448.0           # 1.75 * 2**8
E4M3_EMAX = 8              # exponent of the largest normal power of two
E4M3_NAN = 0x7F


def e4m3_decode(code) -> np.ndarray:
    """Value of E4M3 codes by the format's definition (bias 7, subnormals, S.1111.111 = NaN)."""
    c = np.asarray(code).astype(np.int64)
    s = (c >> 7) & 1
    E = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(E == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, E - 7))
    val = np.where((E == 15) & (m == 7), np.nan, val)
    return np.where(s == 1, -val, val)


def e4m3_rne_satfinite(q) -> np.ndarray:
    """RNE float64 -> E4M3 code, magnitudes beyond 448 saturate to 448.

    The value is rounded on the E4M3 grid (3 fraction bits, smallest normal exponent
    -6, subnormal spacing 2**-9) and then clamped; sign is kept (negative values that
    round to zero give -0 = 0x80).  NaN input gives 0x7F.
    """
    q = np.asarray(q, dtype=np.float64)
    fin = np.isfinite(q)
    r = _round_to_grid_rne(np.where(fin, q, 0.0), frac_bits=3, min_exp=-6)
    r = np.where(np.abs(r) > E4M3_MAX, np.copysign(E4M3_MAX, r), r)
    r = np.where(np.isinf(q), np.copysign(E4M3_MAX, q), r)
    a = np.abs(r)
    sign = np.signbit(np.where(fin | np.isinf(q), r, 0.0)).astype(np.int64)
    with np.errstate(divide="ignore"):
        _, e = np.frexp(a)
    exp = e - 1                                     # floor(log2 a) for a > 0
    normal = a >= 2.0 ** -6
    E = np.where(normal, exp + 7, 0)
    mant = np.where(normal, np.ldexp(a, -exp) - 1.0, a / 2.0 ** -6)   # exact fractions of 1/8
    m = np.rint(mant * 8.0).astype(np.int64)
    code = (sign << 7) | (E.astype(np.int64) << 3) | m
    code = np.where(np.isnan(q), E4M3_NAN, code)
    return code.astype(np.uint8)


# ----------------------------------------------------------------------------- E2M1

E2M1_MAX = 6.0             # 1.5 * 2**2


def e2m1_decode(code) -> np.ndarray:
    """Value of 4-bit E2M1 codes by the format's definition: 1 sign, 2 exponent (bias 1),
    1 mantissa bit, subnormals (exponent field 0: m * 0.5), no infinity and no NaN."""
    c = np.asarray(code).astype(np.int64) & 0xF
    s = (c >> 3) & 1
    E = (c >> 1) & 0x3
    m = c & 0x1
    val = np.where(E == 0, m * 0.5, (1.0 + m / 2.0) * np.ldexp(1.0, E - 1))
    return np.where(s == 1, -val, val)


def e2m1_rne_satfinite(q) -> np.ndarray:
    """RNE float64 -> E2M1 code (0..15), magnitudes beyond 6 saturate to 6.

    Rounded on the E2M1 grid (1 fraction bit, smallest normal exponent 0, subnormal
    spacing 0.5), then clamped; the sign is kept (-0 = 0x8).  Finite input only."""
    q = np.asarray(q, dtype=np.float64)
    r = _round_to_grid_rne(q, frac_bits=1, min_exp=0)
    r = np.where(np.abs(r) > E2M1_MAX, np.copysign(E2M1_MAX, r), r)
    a = np.abs(r)
    sign = np.signbit(r).astype(np.int64)
    with np.errstate(divide="ignore"):
        _, e = np.frexp(a)
    exp = e - 1                                     # floor(log2 a) for a > 0
    normal = a >= 1.0
    E = np.where(normal, exp + 1, 0)
    # normal: a = (1 + m/2) 2**exp; subnormal: a = m * 0.5 (both exact halves)
    m = np.where(normal, np.rint((np.ldexp(a, -exp) - 1.0) * 2.0), np.rint(a * 2.0)).astype(np.int64)
    return ((sign << 3) | (E.astype(np.int64) << 1) | m).astype(np.uint8)


# ----------------------------------------------------------------------------- E8M0

def e8m0_value(byte) -> np.ndarray:
    b = np.asarray(byte).astype(np.int64)
    v = np.ldexp(1.0, b - 127)
    return np.where(b == 0xFF, np.nan, v)
