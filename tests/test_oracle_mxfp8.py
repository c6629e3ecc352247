"""Pins of the MXFP8 oracle: the scale rule in closed form, exhaustive nearest-code search,
the error bound, special blocks, the page's bytes-per-element table, and the GEMM."""
import numpy as np
import pytest

from oracle import floats as F
from oracle import gemm as G
from oracle import mxfp8 as MX


def test_scale_exponent_closed_form():
    """amax in [2^k, 2^(k+1)) -> scale 2^(k-8), so amax / scale lies in [256, 512)."""
    for k in range(-118, 128):
        for frac in (1.0, 1.37, 1.9999):
            a = np.float32(frac * 2.0 ** k)
            if not np.isfinite(a) or a == 0:
                continue
            e = MX.block_scale_exponent(np.array([a], np.float32))[0]
            assert e == k - 8
            assert 256 <= float(a) / 2.0 ** e < 512
    # zero, fp32 subnormals and tiny normals clamp to 2^-127
    for a in (0.0, 1e-45, 1e-40, 2.0 ** -126, 2.0 ** -119):
        assert MX.block_scale_exponent(np.array([a], np.float32))[0] == -127


def brute_force_code(x: float, e: int) -> int:
    """The E4M3 code nearest to x / 2^e among all finite codes; ties to even mantissa; saturate."""
    codes = np.arange(256)
    vals = F.e4m3_decode(codes)
    ok = ~np.isnan(vals)
    q = x / 2.0 ** e
    if abs(q) > 448:
        return 0x7E | (0x80 if q < 0 else 0)
    d = np.abs(vals[ok] - q)
    best = np.flatnonzero(d == d.min())
    cands = codes[ok][best]
    # among equally near codes of the right sign, prefer an even mantissa (then the sign of q)
    cands = sorted(cands, key=lambda c: ((c & 1), (c >> 7) != (1 if np.signbit(q) else 0)))
    return int(cands[0])


def test_quantize_against_exhaustive_search():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((4, 64)) * np.array([[1e-3], [0.02], [1.0], [300.0]])).astype(np.float32)
    x[0, :32] = 0.0
    x[1, 3] = 0.0
    codes, scales = MX.quantize_rowwise(x)
    for r in range(4):
        for b in range(2):
            e = int(scales[r, b]) - 127
            for j in range(32):
                c = b * 32 + j
                want = brute_force_code(float(x[r, c]), e)
                got = int(codes[r, c])
                if x[r, c] == 0:
                    assert got & 0x7F == 0
                else:
                    assert got == want, (r, c, got, want)


def test_error_bound_and_saturation():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    codes, scales = MX.quantize_rowwise(x)
    dq = MX.dequantize_rowwise(codes, scales)
    s = np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)
    q = x / s
    _, ex = np.frexp(np.abs(q))
    ulp = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)       # E4M3 spacing at |q|
    sat = np.abs(q) > 448
    err = np.abs(dq - x)
    assert np.all(err[~sat] <= 0.5 * ulp[~sat] * s[~sat] * (1 + 1e-12))
    assert np.all(np.abs(dq[sat]) == 448 * s[sat])
    assert np.all(err[sat] <= 64 * s[sat])
    # amax of each block maps into [256, 512) before rounding
    amax = np.abs(x).reshape(64, 8, 32).max(axis=2)
    assert np.all((amax / np.ldexp(1.0, scales.astype(np.int64) - 127) >= 256)
                  & (amax / np.ldexp(1.0, scales.astype(np.int64) - 127) < 512))


def test_special_blocks():
    x = np.zeros((3, 64), np.float32)
    x[1, 5] = np.nan
    x[2, 40] = -np.inf
    x[2, 0] = 1.0
    codes, scales = MX.quantize_rowwise(x)
    assert scales[0, 0] == 0 and not codes[0].any()
    assert scales[1, 0] == 0xFF and np.all(codes[1, :32] == 0x7F) and scales[1, 1] == 0
    assert scales[2, 1] == 0xFF and np.all(codes[2, 32:] == 0x7F)
    assert scales[2, 0] == 127 - 8 and codes[2, 0] == 0x78          # 1.0 -> 256 = 1.0 * 2^8
    with pytest.raises(ValueError):
        MX.quantize_rowwise(np.zeros((2, 48), np.float32))


def test_block_format_matches_page_table(golden):
    """[GTP] §1.3 table: block 32, 1 + 1/32 bytes per element, totals per microbatch."""
    g = golden("mx_block_format.json")["MXFP8"]
    R, C = 8, 256
    codes, scales = MX.quantize_rowwise(np.ones((R, C), np.float32))
    assert scales.shape == (R, C // g["block"])
    per_elem = (codes.nbytes + scales.nbytes) / (R * C)
    assert per_elem == 1 + 1 / 32
    # the page prints four decimals, rounding half up (1.03125 -> 1.0313)
    assert abs(per_elem - g["per_elem_printed"]) <= 5.001e-5
    assert abs(1 / 32 - g["scale_bytes_per_elem_printed"]) <= 5.001e-5
    assert abs(2 * per_elem + 2.0 - g["total_printed"]) < 2e-4
    nv = golden("mx_block_format.json")["NVFP4"]
    assert 0.5 + 1 / nv["block"] == nv["per_elem_printed"] and 2 * 0.5625 + 2 == nv["total_printed"]


def test_bf16_source_equals_fp32_source():
    rng = np.random.default_rng(2)
    xb = F.f32_to_bf16_bits(rng.standard_normal((16, 64)).astype(np.float32))
    a = MX.quantize_rowwise(xb, src_is_bf16_bits=True)
    b = MX.quantize_rowwise(F.bf16_bits_to_f32(xb))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_columnwise_view_blocks_run_down_columns():
    """Each scale of the columnwise view is the closed-form exponent of a 32-row block of one
    column, and its codes dequantize back within the block error bound."""
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((96, 5)) * np.exp2(rng.integers(-5, 5, size=(1, 5)))).astype(np.float32)
    qt, st = MX.quantize_columnwise(x)
    assert qt.shape == (5, 96) and st.shape == (5, 3)
    for c in range(5):
        for rb in range(3):
            blk = x[32 * rb:32 * rb + 32, c]
            e = MX.block_scale_exponent(np.array([np.abs(blk).max()], np.float32))[0]
            assert st[c, rb] == e + 127
    # codes of a column block are those of the same 32 values quantized as one row block
    for c in range(5):
        for rb in range(3):
            q1, s1 = MX.quantize_rowwise(x[32 * rb:32 * rb + 32, c][None, :].copy())
            assert np.array_equal(qt[c, 32 * rb:32 * rb + 32], q1[0]) and st[c, rb] == s1[0, 0]


def test_backward_products_are_the_transposed_forward():
    rng = np.random.default_rng(9)
    dY = rng.standard_normal((64, 32)).astype(np.float32)
    Wt = (rng.standard_normal((32, 96)) * 0.02).astype(np.float32)
    dq, ds = MX.quantize_rowwise(dY)
    wq, ws = MX.quantize_columnwise(Wt)
    np.testing.assert_allclose(MX.dgrad_mxfp8(dq, ds, wq, ws),
                               MX.dequantize_rowwise(dq, ds) @ MX.dequantize_rowwise(wq, ws).T, rtol=0, atol=0)
    X = rng.standard_normal((64, 96)).astype(np.float32)
    dtq, dts = MX.quantize_columnwise(dY)
    xq, xs = MX.quantize_columnwise(X)
    G = MX.wgrad_accum_mxfp8(np.zeros((32, 96), np.float32), dtq, dts, xq, xs)
    ref = (MX.dequantize_rowwise(dtq, dts) @ MX.dequantize_rowwise(xq, xs).T).astype(np.float32)
    assert np.array_equal(G, ref)


def test_flat_blocks_are_each_weights_rowwise_view():
    """A flat buffer of weights at 64-aligned offsets (the dist-opt layout) with zero padding
    between them: each weight's slice of the flat-block quantization is its rowwise view,
    and padding blocks are scale 0 / code 0."""
    rng = np.random.default_rng(10)
    shapes = [(7, 96), (3, 32), (5, 160)]
    buf = np.zeros(2048, np.float32)
    offs, cur = [], 0
    for (n, k) in shapes:
        cur = -(-cur // 64) * 64
        offs.append(cur)
        buf[cur:cur + n * k] = (rng.standard_normal(n * k) * np.exp2(rng.integers(-8, 8, size=n * k))).astype(np.float32)
        cur += n * k
    codes, scales = MX.quantize_flat_blocks(buf)
    assert codes.shape == (2048,) and scales.shape == (64,)
    covered = np.zeros(2048, bool)
    for (n, k), o in zip(shapes, offs):
        q, s = MX.quantize_rowwise(buf[o:o + n * k].reshape(n, k))
        assert np.array_equal(codes[o:o + n * k], q.reshape(-1))
        assert np.array_equal(scales[o // 32:(o + n * k) // 32], s.reshape(-1))
        covered[o:o + n * k] = True
    assert not codes[~covered].any()
    assert not scales[~covered.reshape(-1, 32).any(axis=1)].any()
    with pytest.raises(ValueError):
        MX.quantize_flat_blocks(np.zeros(48, np.float32))


def test_fprop_on_dequantized_operands():
    rng = np.random.default_rng(3)
    X = rng.standard_normal((6, 64)).astype(np.float32)
    Wt = (rng.standard_normal((5, 64)) * 0.02).astype(np.float32)
    Xq, Xs = MX.quantize_rowwise(X)
    Wq, Ws = MX.quantize_rowwise(Wt)
    Y = MX.fprop_mxfp8(Xq, Xs, Wq, Ws)
    Xd = MX.dequantize_rowwise(Xq, Xs).tolist()
    Wd = MX.dequantize_rowwise(Wq, Ws).tolist()
    np.testing.assert_allclose(Y, np.array(G.matmul_loops(Xd, G.transpose_loops(Wd))), rtol=1e-14, atol=1e-14)
    assert MX.fprop_mxfp8_bf16(Xq, Xs, Wq, Ws).dtype == np.uint16
