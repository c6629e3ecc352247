"""MXFP8 weight quantize and the MXFP8 forward GEMM (oracle; test infrastructure).

[GTP] §1.3: native MXFP8 weights are written from the fp32 master once per optimizer
step, off the forward critical path; the rowwise view serves the forward GEMM.  The
format is "Block 32", with 1/32 byte of scale per element (table "Communication volume
breakdown"): one scale byte per 32-element block next to one byte per element.

Reading R5 (the pages name neither the element format nor the scale rule): elements
are E4M3, scales E8M0, and the scale of a block follows the OCP Microscaling (MX) v1.0
rule: X = 2**(floor(log2(amax)) - emax_elem) with emax_elem = 8 for E4M3, clamped to
the E8M0 range; each element becomes RNE_E4M3(x / X), saturating at +-448.
Special cases: amax == 0 gives scale byte 0 (2**-127) and zero elements; a block with
any NaN or infinity gives scale 0xFF (NaN) and elements 0x7F.

Reading R6: the forward GEMM consumes both operands in MX form, each quantized
rowwise along the contraction dimension K (blocks of 32 consecutive K elements):
Y = bf16( sum_k dq(Xq)[m, k] * dq(Wq)[n, k] ).
"""
from __future__ import annotations

import numpy as np

from .floats import E4M3_EMAX, E4M3_NAN, bf16_bits_to_f32, e4m3_decode, e4m3_rne_satfinite, f32_bits, f64_to_bf16_bits

BLOCK = 32


def block_scale_exponent(amax_f32: np.ndarray) -> np.ndarray:
    """floor(log2(amax)) - 8, clamped to [-127, 127], from the fp32 encoding of amax.

    For a normal fp32 amax, floor(log2) is its unbiased exponent.  Zero and fp32
    subnormals lie below 2**-126, so the clamped result is -127 for them.
    """
    biased = ((f32_bits(amax_f32) >> np.uint32(23)) & np.uint32(0xFF)).astype(np.int64)
    e = np.where(biased == 0, -127, biased - 127 - E4M3_EMAX)
    return np.clip(e, -127, 127)


def quantize_rowwise(x, src_is_bf16_bits: bool = False):
    """MX-quantize a [R, C] matrix along rows in blocks of 32: (e4m3 [R,C], e8m0 [R,C/32])."""
    if src_is_bf16_bits:
        x = bf16_bits_to_f32(x)
    x = np.asarray(x, dtype=np.float32)
    R, C = x.shape
    if C % BLOCK:
        raise ValueError("columns must be a multiple of 32")
    xb = x.reshape(R, C // BLOCK, BLOCK)
    finite = np.all(np.isfinite(xb), axis=2)
    amax = np.max(np.abs(np.where(np.isfinite(xb), xb, 0)), axis=2).astype(np.float32)
    e = block_scale_exponent(amax)
    scale = (e + 127).astype(np.int64)
    q = np.ldexp(xb.astype(np.float64), -e[:, :, None])     # exact power-of-two scaling
    codes = e4m3_rne_satfinite(q)
    codes = np.where(finite[:, :, None], codes, E4M3_NAN).astype(np.uint8)
    scale = np.where(finite, scale, 0xFF).astype(np.uint8)
    return codes.reshape(R, C), scale


def dequantize_rowwise(codes, scales) -> np.ndarray:
    R, C = codes.shape
    v = e4m3_decode(codes).reshape(R, C // BLOCK, BLOCK)
    s = scales.astype(np.int64)
    out = np.ldexp(v, (s - 127)[:, :, None])
    out = np.where((s == 0xFF)[:, :, None], np.nan, out)
    return out.reshape(R, C)


def fprop_mxfp8(Xq, Xs, Wq, Ws) -> np.ndarray:
    """Y = dq(Xq) dq(Wq)^T in float64 (exact products; reading R6)."""
    return dequantize_rowwise(Xq, Xs) @ dequantize_rowwise(Wq, Ws).T


def fprop_mxfp8_bf16(Xq, Xs, Wq, Ws) -> np.ndarray:
    return f64_to_bf16_bits(fprop_mxfp8(Xq, Xs, Wq, Ws))


def quantize_flat_blocks(x):
    """MX blocks of 32 consecutive elements of a flat buffer (numel % 32 == 0): the
    rowwise rule on x viewed as [numel/32, 32].  For a weight [N, K] stored at an offset
    that is a multiple of 32 with K % 32 == 0, its slice of the result is its rowwise view
    (the native MXFP8 parameter buffer of [GTP] §1.3)."""
    x = np.asarray(x, dtype=np.float32).reshape(-1)
    if x.size % BLOCK:
        raise ValueError("numel must be a multiple of 32")
    codes, scales = quantize_rowwise(x.reshape(-1, BLOCK))
    return codes.reshape(-1), scales.reshape(-1)


def quantize_columnwise(x, src_is_bf16_bits: bool = False):
    """The columnwise (backward) view of [GTP] §1.3: 32-element blocks down each column,
    stored transposed - by definition the rowwise quantization of x^T (reading R14)."""
    return quantize_rowwise(np.ascontiguousarray(np.asarray(x).T), src_is_bf16_bits=src_is_bf16_bits)


def dgrad_mxfp8(dYq, dYs, Wtq, Wts) -> np.ndarray:
    """dX = dq(dY) dq(W^T)^T in float64 (contraction over N)."""
    return dequantize_rowwise(dYq, dYs) @ dequantize_rowwise(Wtq, Wts).T


def wgrad_accum_mxfp8(main_grad_f32, dYtq, dYts, Xtq, Xts) -> np.ndarray:
    """main_grad <- fp32(main_grad + dq(dY^T) dq(X^T)^T) (contraction over tokens M)."""
    acc = main_grad_f32.astype(np.float64) + dequantize_rowwise(dYtq, dYts) @ dequantize_rowwise(Xtq, Xts).T
    return acc.astype(np.float32)
