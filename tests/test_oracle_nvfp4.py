"""Pins of the NVFP4 oracle: the E2M1 format from its bit definition and by exhaustive
nearest-value search, the two-level scale rule in closed form, the error bound, special
tensors, the page's bytes-per-element table, and the GEMM against triple loops."""
import numpy as np
import pytest

from oracle import floats as F
from oracle import gemm as G
from oracle import nvfp4 as NV

E2M1_MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]    # the format's eight magnitudes


def test_e2m1_decode_table():
    vals = F.e2m1_decode(np.arange(16))
    assert list(vals[:8]) == E2M1_MAGS
    assert list(-vals[8:]) == E2M1_MAGS and np.signbit(vals[8])


def brute_e2m1(q: float) -> int:
    """Nearest of the 16 codes, ties to the even mantissa bit, saturating at 6."""
    codes = np.arange(16)
    vals = F.e2m1_decode(codes)
    if abs(q) > 6:
        return 0x7 | (0x8 if q < 0 else 0)
    d = np.abs(vals - q)
    cands = codes[d == d.min()]
    sign = 1 if np.signbit(q) else 0
    cands = sorted(cands, key=lambda c: ((c & 1), (c >> 3) != sign))
    return int(cands[0])


def test_e2m1_rounding_exhaustive():
    grid = np.unique(np.concatenate([np.linspace(-8, 8, 4097),
                                     np.array(E2M1_MAGS) + 0.0, -np.array(E2M1_MAGS),
                                     [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 6.5, 7.0, 1e-30, -1e-30]]))
    got = F.e2m1_rne_satfinite(grid)
    for q, c in zip(grid, got):
        assert int(c) == brute_e2m1(float(q)), (q, c)
    # the ties by hand: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    ties = F.e2m1_decode(F.e2m1_rne_satfinite(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])))
    assert list(ties) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_tensor_scale_closed_form():
    assert NV.tensor_scale(0.0) == 1.0
    assert NV.tensor_scale(2688.0) == 1.0
    assert NV.tensor_scale(1.0) == np.float32(2688.0)
    assert NV.tensor_scale(1e-40) == np.finfo(np.float32).max          # clamped
    # the block holding the tensor amax gets the largest scale, 448 = code 0x7E, when the
    # fp32 steps are exact (amax a power of two times 6)
    x = np.zeros((2, 32), np.float32)
    x[1, 20] = 6.0 * 2.0 ** -3
    x[0, :16] = 0.01
    _, sf, A = NV.quantize_rowwise(x)
    assert A == np.float32(0.75) and sf[1, 1] == 0x7E


def test_constant_block_maps_to_six():
    """A block of one value c: every code is +-6 and the dequantized block is within the
    E4M3 scale's relative rounding (2^-4) of c."""
    rng = np.random.default_rng(0)
    for c in rng.standard_normal(50) * np.exp2(rng.integers(-20, 20, size=50)):
        x = np.full((1, 16), np.float32(c), np.float32)
        x = np.concatenate([x, np.full((1, 16), np.float32(abs(c) * 3), np.float32)])   # sets the tensor amax
        p, sf, A = NV.quantize_rowwise(x)
        codes = NV.unpack(p)[0]
        assert np.all(codes == (0x7 | (0x8 if c < 0 else 0)))
        dq = NV.dequantize_rowwise(p, sf, A)[0]
        assert np.all(np.abs(dq - np.float32(c)) <= abs(float(np.float32(c))) / 16 * (1 + 1e-9))


def test_error_bound():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    p, sf, A = NV.quantize_rowwise(x)
    dq = NV.dequantize_rowwise(p, sf, A)
    S = float(NV.tensor_scale(A))
    s = np.repeat(F.e4m3_decode(sf), 16, axis=1) / S                      # the element step scale
    q = np.abs(x) / s
    half = np.where(q < 2, 0.25, np.where(q < 4, 0.5, 1.0))              # half the E2M1 spacing
    sat = q > 6
    err = np.abs(dq - x)
    assert np.all(err[~sat] <= half[~sat] * s[~sat] * (1 + 1e-6))
    np.testing.assert_allclose(np.abs(dq[sat]), 6 * s[sat], rtol=1e-12)
    assert np.all(q <= 6 * (1 + 2.0 ** -4) * (1 + 1e-6))                # the scale rounds by <= 2^-4


def test_special_tensors():
    p, sf, A = NV.quantize_rowwise(np.zeros((2, 32), np.float32))
    assert A == 0 and not p.any() and not sf.any()
    x = np.ones((2, 32), np.float32)
    x[0, 3] = np.nan
    x[1, 31] = -np.inf
    p, sf, A = NV.quantize_rowwise(x)
    assert A == 1.0
    assert sf[0, 0] == 0x7F and sf[0, 1] != 0x7F and sf[1, 1] == 0x7F and sf[1, 0] != 0x7F
    assert not NV.unpack(p)[0, :16].any() and not NV.unpack(p)[1, 16:].any()
    assert np.all(np.isnan(NV.dequantize_rowwise(p, sf, A)[0, :16]))
    # a tensor of fp32 subnormals: S clamps to FLT_MAX, S / sf overflows and clamps too, so
    # zeros stay zero codes (never 0 * inf) and the dequantized values stay finite
    x = np.zeros((1, 16), np.float32)
    x[0, 1:] = np.float32(1e-40)
    p, sf, A = NV.quantize_rowwise(x)
    assert NV.tensor_scale(A) == np.finfo(np.float32).max and sf[0, 0] != 0
    codes = NV.unpack(p)[0]
    assert codes[0] == 0 and np.all(np.isfinite(NV.dequantize_rowwise(p, sf, A)))
    with pytest.raises(ValueError):
        NV.quantize_rowwise(np.zeros((2, 24), np.float32))


def test_packing_low_nibble_first():
    x = np.array([[0.5, 6.0] + [0.0] * 14], np.float32) * np.float32(1.0)
    p, sf, A = NV.quantize_rowwise(x)
    # amax 6 -> S = 448, block d = 448 -> sf 448: element scale 1, codes 0.5 -> 1, 6 -> 7
    assert sf[0, 0] == 0x7E and p[0, 0] == (0x1 | (0x7 << 4))


def test_block_format_matches_page_table(golden):
    """[GTP] §1.3 table: NVFP4 block 16, 0.5 + 1/16 = 0.5625 bytes per element."""
    g = golden("mx_block_format.json")["NVFP4"]
    p, sf, _ = NV.quantize_rowwise(np.ones((8, 256), np.float32))
    assert sf.shape == (8, 256 // g["block"])
    per_elem = (p.nbytes + sf.nbytes) / (8 * 256)
    assert per_elem == g["data_bytes_per_elem"] + 1 / 16 == g["per_elem_printed"]


def test_bf16_source_equals_fp32_source():
    rng = np.random.default_rng(2)
    xb = F.f32_to_bf16_bits(rng.standard_normal((16, 64)).astype(np.float32))
    a = NV.quantize_rowwise(xb, src_is_bf16_bits=True)
    b = NV.quantize_rowwise(F.bf16_bits_to_f32(xb))
    assert all(np.array_equal(u, v) for u, v in zip(a, b))


def test_fprop_on_dequantized_operands():
    rng = np.random.default_rng(3)
    X = rng.standard_normal((6, 64)).astype(np.float32)
    Wt = (rng.standard_normal((5, 64)) * 0.02).astype(np.float32)
    Xq, Xs, xa = NV.quantize_rowwise(X)
    Wq, Ws, wa = NV.quantize_rowwise(Wt)
    Y = NV.fprop_nvfp4(Xq, Xs, xa, Wq, Ws, wa)
    Xd = NV.dequantize_rowwise(Xq, Xs, xa).tolist()
    Wd = NV.dequantize_rowwise(Wq, Ws, wa).tolist()
    np.testing.assert_allclose(Y, np.array(G.matmul_loops(Xd, G.transpose_loops(Wd))), rtol=1e-14, atol=1e-14)
    assert NV.fprop_nvfp4_bf16(Xq, Xs, xa, Wq, Ws, wa).dtype == np.uint16
    # the quantized product is close to the exact one (4-bit elements: a few percent)
    exact = X.astype(np.float64) @ Wt.astype(np.float64).T
    assert np.linalg.norm(Y - exact) / np.linalg.norm(exact) < 0.2
