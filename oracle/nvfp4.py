"""NVFP4 weight quantize and the NVFP4 forward GEMM (oracle; test infrastructure).

[GTP] §1.3 and its "GTP + NVFP4" subsection: a native NVFP4 parameter is kept as packed
4-bit E2M1 elements (kFloat4E2M1), written by the optimizer once per step, with its
per-tensor scale "set at opt-step quantize"; the table "Communication volume breakdown"
gives block 16 with 1/16 byte of scale per element, 0.5625 bytes per element in all.
[BUF] §5 (special layouts): the NVFP4 param buffer holds the packed bytes, numel / 2.

Reading R16 (the pages name the element format, the block size and the per-tensor scale,
but not the scale rule): the two-level rule of NVIDIA's NVFP4 recipe, every step in fp32.
  A   = max |x| over the finite elements of the tensor (fp32)
  S   = 1 if A == 0, else min(fp32(2688 / A), FLT_MAX)        2688 = 448 * 6
  per block b of 16 consecutive elements of a row, amax_b = max |x| over the block:
  d_b  = fp32(fp32(amax_b / 6) * S);  sf_b = RNE_E4M3_satfinite(d_b)  (one byte, >= 0)
  e_b  = min(fp32(S / value(sf_b)), FLT_MAX), or 0 when value(sf_b) == 0
  code = RNE_E2M1_satfinite(fp32(x * e_b))           (the sign of zero kept: -0 = 0x8)
  dequantized x = e2m1(code) * value(sf_b) / S
A block holding NaN or Inf gets scale byte 0x7F (E4M3 NaN) and codes 0.  Two codes share
a byte, the even element in the low nibble.  The forward GEMM consumes both operands in
this form, quantized along K: Y = bf16( sum_k dq(Xq)[m, k] * dq(Wq)[n, k] ).
"""
from __future__ import annotations

import numpy as np

from .floats import bf16_bits_to_f32, e2m1_decode, e2m1_rne_satfinite, e4m3_decode, e4m3_rne_satfinite, f64_to_bf16_bits

BLOCK = 16
E4M3_X_E2M1 = np.float32(448.0 * 6.0)
FLT_MAX = np.float32(np.finfo(np.float32).max)
SCALE_NAN = 0x7F


def tensor_amax(x) -> np.float32:
    x = np.asarray(x, dtype=np.float32)
    fin = np.isfinite(x)
    return np.float32(np.max(np.abs(x[fin]))) if fin.any() else np.float32(0.0)


def tensor_scale(amax) -> np.float32:
    """S of reading R16 from the fp32 tensor amax."""
    a = np.float32(amax)
    if a == 0:
        return np.float32(1.0)
    with np.errstate(over="ignore", divide="ignore"):
        s = np.float32(E4M3_X_E2M1 / a)
    return np.float32(min(s, FLT_MAX))


def quantize_rowwise(x, src_is_bf16_bits: bool = False, amax=None):
    """[R, C] -> (packed uint8 [R, C/2], e4m3 scales [R, C/16], tensor amax fp32).

    ``amax`` defaults to the tensor's own (reading R16); the columns must be a multiple
    of 16."""
    if src_is_bf16_bits:
        x = bf16_bits_to_f32(x)
    x = np.asarray(x, dtype=np.float32)
    R, C = x.shape
    if C % BLOCK:
        raise ValueError("columns must be a multiple of 16")
    A = tensor_amax(x) if amax is None else np.float32(amax)
    S = tensor_scale(A)
    xb = x.reshape(R, C // BLOCK, BLOCK)
    finite = np.all(np.isfinite(xb), axis=2)
    amax_b = np.max(np.abs(np.where(np.isfinite(xb), xb, 0)), axis=2).astype(np.float32)
    with np.errstate(over="ignore"):
        d = ((amax_b / np.float32(6.0)).astype(np.float32) * S).astype(np.float32)
    sf = e4m3_rne_satfinite(d.astype(np.float64))
    sfv = e4m3_decode(sf).astype(np.float32)                    # exact in fp32
    with np.errstate(divide="ignore", over="ignore"):
        ratio = (S / np.where(sfv == 0, np.float32(1.0), sfv)).astype(np.float32)
        enc = np.where(sfv == 0, np.float32(0.0), np.minimum(ratio, FLT_MAX)).astype(np.float32)
        q = (np.where(np.isfinite(xb), xb, 0).astype(np.float32) * enc[:, :, None]).astype(np.float32)
    codes = e2m1_rne_satfinite(q.astype(np.float64)).astype(np.uint8)
    codes = np.where(finite[:, :, None], codes, 0).astype(np.uint8).reshape(R, C)
    sf = np.where(finite, sf, SCALE_NAN).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, sf, np.float32(A)


def unpack(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


def dequantize_rowwise(packed, scales, amax) -> np.ndarray:
    codes = unpack(packed)
    R, C = codes.shape
    v = e2m1_decode(codes).reshape(R, C // BLOCK, BLOCK)
    s = e4m3_decode(scales)                                    # NaN for 0x7F
    out = v * s[:, :, None] / np.float64(tensor_scale(amax))
    return out.reshape(R, C)


def fprop_nvfp4(Xq, Xs, x_amax, Wq, Ws, w_amax) -> np.ndarray:
    """Y = dq(Xq) dq(Wq)^T in float64."""
    return dequantize_rowwise(Xq, Xs, x_amax) @ dequantize_rowwise(Wq, Ws, w_amax).T


def fprop_nvfp4_bf16(Xq, Xs, x_amax, Wq, Ws, w_amax) -> np.ndarray:
    return f64_to_bf16_bits(fprop_nvfp4(Xq, Xs, x_amax, Wq, Ws, w_amax))
