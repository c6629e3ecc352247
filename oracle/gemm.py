"""The three GEMMs of the tensor-parallel linear layer (oracle; test infrastructure).

[LIN] §4.1 (forward): ``output = total_input @ weight.t()``, the weight of one TP
shard stored [out, in] ([LIN] §1: column-parallel [out/TP, in], row-parallel
[out, in/TP]).

[LIN] §4.2 (backward): dgrad ``grad_input = grad_output @ weight``; wgrad with
gradient_accumulation_fusion accumulates ``grad_output^T @ total_input`` straight into
the fp32 ``weight.main_grad``, which is a view of the flat grad buffer
([BUF] §5: ``param.main_grad = grad_data[s:e].view(shape)``).

Notation: M tokens (s*b), N out-features, K in-features of the shard; X [M, K],
W [N, K], Y / dY [M, N], dX [M, K], main_grad [N, K]; all row-major.

The products are exact definitions evaluated in float64 from the exact float64 values
of the bf16 inputs.  Reading R2: the in-place fp32 main_grad is rounded to fp32 once
per accumulate call (one microbatch), as an fp32 tensor updated in place is.
"""
from __future__ import annotations

import numpy as np

from .floats import bf16_bits_to_f64, f64_to_bf16_bits


def fprop(X_bf16: np.ndarray, W_bf16: np.ndarray) -> np.ndarray:
    """Y = X W^T in float64 (X [M,K], W [N,K] as bf16 bit patterns)."""
    return bf16_bits_to_f64(X_bf16) @ bf16_bits_to_f64(W_bf16).T


def dgrad(dY_bf16: np.ndarray, W_bf16: np.ndarray) -> np.ndarray:
    """dX = dY W in float64 (dY [M,N], W [N,K])."""
    return bf16_bits_to_f64(dY_bf16) @ bf16_bits_to_f64(W_bf16)


def wgrad(dY_bf16: np.ndarray, X_bf16: np.ndarray) -> np.ndarray:
    """dW = dY^T X in float64 ([N, K])."""
    return bf16_bits_to_f64(dY_bf16).T @ bf16_bits_to_f64(X_bf16)


def wgrad_accum(main_grad_f32: np.ndarray, dY_bf16: np.ndarray, X_bf16: np.ndarray) -> np.ndarray:
    """main_grad <- fp32(main_grad + dY^T X) (one fp32 rounding per call, reading R2)."""
    acc = main_grad_f32.astype(np.float64) + wgrad(dY_bf16, X_bf16)
    return acc.astype(np.float32)


def to_bf16(y: np.ndarray) -> np.ndarray:
    """The bf16 output of fprop / dgrad: one RNE rounding of the exact product."""
    return f64_to_bf16_bits(y)


# ----------------------------------------------------------------------------- brute force

def matmul_loops(A: list, B: list) -> list:
    """C[i][j] = sum_k A[i][k] * B[k][j], written as three loops (tiny shapes only)."""
    m, k = len(A), len(A[0])
    n = len(B[0])
    assert len(B) == k
    C = [[0.0] * n for _ in range(m)]
    for i in range(m):
        for j in range(n):
            s = 0.0
            for t in range(k):
                s += A[i][t] * B[t][j]
            C[i][j] = s
    return C


def transpose_loops(A: list) -> list:
    return [[A[i][j] for i in range(len(A))] for j in range(len(A[0]))]


def sampled_fprop(X_bf16, W_bf16, rows, cols) -> np.ndarray:
    """Y[rows[i], cols[i]] one dot product at a time (for full-size shapes)."""
    X = X_bf16[rows]
    W = W_bf16[cols]
    return np.einsum("ik,ik->i", bf16_bits_to_f64(X), bf16_bits_to_f64(W))


def sampled_dgrad(dY_bf16, W_bf16, rows, cols) -> np.ndarray:
    """dX[rows[i], cols[i]] = sum_n dY[rows[i], n] W[n, cols[i]]."""
    dY = bf16_bits_to_f64(dY_bf16[rows])
    Wc = bf16_bits_to_f64(W_bf16[:, cols]).T
    return np.einsum("in,in->i", dY, Wc)


def sampled_wgrad(dY_bf16, X_bf16, rows, cols) -> np.ndarray:
    """dW[rows[i], cols[i]] = sum_m dY[m, rows[i]] X[m, cols[i]]."""
    dYc = bf16_bits_to_f64(dY_bf16[:, rows]).T
    Xc = bf16_bits_to_f64(X_bf16[:, cols]).T
    return np.einsum("im,im->i", dYc, Xc)


def sampled_wgrad_accum(main_grad_at: np.ndarray, dY_bf16, X_bf16, rows, cols) -> np.ndarray:
    """main_grad[rows[i], cols[i]] <- fp32(main_grad[rows[i], cols[i]] + dW[rows[i], cols[i]]):
    wgrad_accum at sampled positions only, with the same single fp32 rounding per call
    (reading R2).  main_grad_at holds the fp32 values at those positions."""
    acc = np.asarray(main_grad_at, np.float32).astype(np.float64) + sampled_wgrad(dY_bf16, X_bf16, rows, cols)
    return acc.astype(np.float32)


def wgrad_accum_bf16(main_grad_bf16: np.ndarray, dY_bf16: np.ndarray, X_bf16: np.ndarray) -> np.ndarray:
    """A bf16 main_grad (grad_reduce_in_fp32 off: the BufferKey's grad dtype is the
    parameter's, [BUF] §3) accumulated in high precision and stored as bf16 (reading R18):
    main_grad <- RNE_bf16(main_grad + dY^T X), one rounding of the exact sum per call.
    Bit patterns in, bit patterns out."""
    return f64_to_bf16_bits(bf16_bits_to_f64(main_grad_bf16) + wgrad(dY_bf16, X_bf16))


def sampled_wgrad_accum_bf16(main_grad_at_bf16, dY_bf16, X_bf16, rows, cols) -> np.ndarray:
    """wgrad_accum_bf16 at sampled positions (bf16 bit patterns of main_grad there)."""
    return f64_to_bf16_bits(bf16_bits_to_f64(np.asarray(main_grad_at_bf16, np.uint16))
                            + sampled_wgrad(dY_bf16, X_bf16, rows, cols))
