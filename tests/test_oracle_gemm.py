"""Pins of the GEMM oracle: a triple loop on tiny shapes, closed forms, and the sampled
single-dot-product forms used at full size."""
import numpy as np
import torch

from oracle import floats as F
from oracle import gemm as G
from param_buffers_gb300 import workloads as W


def bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).numpy().view(np.uint16)


def tiny_inputs(M=5, N=4, K=3, seed=0):
    g = W.generator(seed)
    X, Wt, dY = W.linear_inputs(M, N, K, g, w_std=0.5)
    return bits(X), bits(Wt), bits(dY)


def to_list(a):
    return [[float(v) for v in row] for row in a]


def test_fprop_dgrad_wgrad_against_loops():
    X, Wt, dY = tiny_inputs()
    Xf, Wf, dYf = (to_list(F.bf16_bits_to_f64(a)) for a in (X, Wt, dY))
    np.testing.assert_array_equal(G.fprop(X, Wt), np.array(G.matmul_loops(Xf, G.transpose_loops(Wf))))
    np.testing.assert_array_equal(G.dgrad(dY, Wt), np.array(G.matmul_loops(dYf, Wf)))
    np.testing.assert_array_equal(G.wgrad(dY, X), np.array(G.matmul_loops(G.transpose_loops(dYf), Xf)))


def test_shapes_and_transposes():
    X, Wt, dY = tiny_inputs(7, 6, 5, seed=1)
    assert G.fprop(X, Wt).shape == (7, 6)
    assert G.dgrad(dY, Wt).shape == (7, 5)
    assert G.wgrad(dY, X).shape == (6, 5)
    # dgrad and wgrad are the adjoints of fprop: <dY, X W^T> = <dY W, X> = <dY^T X, W>
    Y = G.fprop(X, Wt)
    Xf, Wf, dYf = (F.bf16_bits_to_f64(a) for a in (X, Wt, dY))
    a = np.sum(dYf * Y)
    assert np.isclose(a, np.sum(G.dgrad(dY, Wt) * Xf), rtol=1e-12)
    assert np.isclose(a, np.sum(G.wgrad(dY, X) * Wf), rtol=1e-12)


def test_identity_and_rank_one():
    one = F.f32_to_bf16_bits(np.eye(8, dtype=np.float32))
    X, _, _ = tiny_inputs(8, 8, 8, seed=2)
    np.testing.assert_array_equal(G.fprop(X, one), F.bf16_bits_to_f64(X))
    ones = F.f32_to_bf16_bits(np.ones((1, 8), np.float32))
    ramp = F.f32_to_bf16_bits(np.arange(6, dtype=np.float32)[None, :])
    # wgrad of a single token (M = 1): dY^T X is the outer product dY[0] x X[0]
    np.testing.assert_array_equal(G.wgrad(ones, ramp), np.outer(np.ones(8), np.arange(6.0)))
    # a row of eight ones dotted with itself
    assert G.fprop(ones, ones).item() == 8.0


def test_wgrad_accumulates_per_call():
    """main_grad after two calls = fp32(fp32(G0 + d1) + d2) (reading R2)."""
    X1, _, dY1 = tiny_inputs(6, 4, 5, seed=3)
    X2, _, dY2 = tiny_inputs(6, 4, 5, seed=4)
    G0 = np.linspace(-1, 1, 20, dtype=np.float32).reshape(4, 5)
    G1 = G.wgrad_accum(G0, dY1, X1)
    G2 = G.wgrad_accum(G1, dY2, X2)
    ref = (G0.astype(np.float64) + G.wgrad(dY1, X1)).astype(np.float32)
    ref = (ref.astype(np.float64) + G.wgrad(dY2, X2)).astype(np.float32)
    assert G2.dtype == np.float32 and np.array_equal(G2, ref)
    # zero main_grad + one call equals the plain product rounded to fp32
    np.testing.assert_array_equal(G.wgrad_accum(np.zeros((4, 5), np.float32), dY1, X1),
                                  G.wgrad(dY1, X1).astype(np.float32))


def test_sampled_forms_equal_full_products():
    X, Wt, dY = tiny_inputs(33, 17, 9, seed=5)
    rng = np.random.default_rng(0)
    r = rng.integers(0, 33, 50); c = rng.integers(0, 17, 50)
    np.testing.assert_array_equal(G.sampled_fprop(X, Wt, r, c), G.fprop(X, Wt)[r, c])
    c2 = rng.integers(0, 9, 50)
    np.testing.assert_allclose(G.sampled_dgrad(dY, Wt, r, c2), G.dgrad(dY, Wt)[r, c2], rtol=1e-14, atol=1e-14)
    r3 = rng.integers(0, 17, 50)
    np.testing.assert_allclose(G.sampled_wgrad(dY, X, r3, c2), G.wgrad(dY, X)[r3, c2], rtol=1e-14, atol=1e-14)


def test_sampled_accumulate_matches_full_accumulate_and_rounds_per_call():
    """The sampled accumulate equals the full accumulate at the sampled positions over
    several calls (integer-valued bf16 inputs: every sum is exact, so the two agree bit for
    bit), and it rounds to fp32 once per call: at 2^24, where the fp32 spacing is 2, two
    calls adding 1 each leave the value at 2^24 (each 2^24 + 1 ties to even), while one
    rounding of the sum would give 2^24 + 2."""
    rng = np.random.default_rng(11)
    M, N, K = 12, 6, 7
    rounds = []
    for _ in range(3):
        X = torch.tensor(rng.integers(-8, 9, (M, K)), dtype=torch.float32).to(torch.bfloat16)
        dY = torch.tensor(rng.integers(-8, 9, (M, N)), dtype=torch.float32).to(torch.bfloat16)
        rounds.append((bits(dY), bits(X)))
    G0 = rng.standard_normal((N, K)).astype(np.float32)
    r = rng.integers(0, N, 30); c = rng.integers(0, K, 30)
    full, samp = G0, G0[r, c]
    for dY, X in rounds:
        full = G.wgrad_accum(full, dY, X)
        samp = G.sampled_wgrad_accum(samp, dY, X, r, c)
    assert samp.dtype == np.float32 and np.array_equal(samp, full[r, c])
    # per-call rounding at 2^24: dY = e_0 (one row of ones in column 0), X = ones -> dW[0, :] = 1
    one_dY = bits(torch.tensor([[1.0, 0.0]]).to(torch.bfloat16))
    one_X = bits(torch.tensor([[1.0, 1.0]]).to(torch.bfloat16))
    g = np.array([2.0 ** 24], np.float32)
    for _ in range(2):
        g = G.sampled_wgrad_accum(g, one_dY, one_X, np.array([0]), np.array([1]))
    assert g[0] == np.float32(2.0 ** 24)


def test_bf16_main_grad_accumulate():
    """The bf16 main_grad accumulate equals torch's own float64 -> bf16 cast of the exact
    sum (an independent rounding routine), its sampled form equals the full one, and it
    rounds once per call: at 256, where the bf16 spacing is 2, two calls adding 1 each
    leave 256 (each 257 ties to even), while one rounding of 258 would keep 258."""
    rng = np.random.default_rng(21)
    M, N, K = 40, 12, 9
    X, _, dY = tiny_inputs(M, N, K, seed=22)
    G0 = torch.tensor(rng.standard_normal((N, K)) * 4).to(torch.bfloat16)
    got = G.wgrad_accum_bf16(bits(G0), dY, X)
    exact = torch.tensor(F.bf16_bits_to_f64(bits(G0)) + G.wgrad(dY, X), dtype=torch.float64)
    np.testing.assert_array_equal(got, bits(exact.to(torch.bfloat16)))
    r, c = rng.integers(0, N, 30), rng.integers(0, K, 30)
    np.testing.assert_array_equal(G.sampled_wgrad_accum_bf16(bits(G0)[r, c], dY, X, r, c), got[r, c])
    one_dY = bits(torch.tensor([[1.0, 0.0]]).to(torch.bfloat16))
    one_X = bits(torch.tensor([[1.0, 1.0]]).to(torch.bfloat16))
    g = bits(torch.tensor([[256.0, 256.0], [0.0, 0.0]]).to(torch.bfloat16))   # dW = [[1, 1], [0, 0]]
    for _ in range(2):
        g = G.wgrad_accum_bf16(g, one_dY, one_X)
    np.testing.assert_array_equal(F.bf16_bits_to_f64(g), [[256.0, 256.0], [0.0, 0.0]])
    assert F.bf16_bits_to_f64(F.f64_to_bf16_bits(np.array([258.0])))[0] == 258.0   # one rounding would keep 258


def test_bf16_output_rounding_budget():
    """The bf16 output rounding alone costs ~1.6e-3 relative Frobenius error on N(0,1) x N(0,0.02)
    data, inside the 2e-3 tolerance the GEMM parity tests use."""
    g = W.generator(9)
    X, Wt, _ = W.linear_inputs(256, 256, 256, g)
    Y = G.fprop(bits(X), bits(Wt))
    Yb = F.bf16_bits_to_f64(G.to_bf16(Y))
    rel = np.linalg.norm(Yb - Y) / np.linalg.norm(Y)
    assert 1.0e-3 < rel < 2e-3
