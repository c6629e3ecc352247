"""Pins of the gradient-norm oracle: torch's clip_grad_norm_ (float64), closed forms."""
import numpy as np
import torch

from oracle import gradnorm as GN


def test_against_torch_clip_grad_norm():
    rng = np.random.default_rng(0)
    grads = [rng.standard_normal(n) * 1e-3 for n in (100, 37, 1000)]
    for max_norm in (1.0, 0.01, 1e-5):
        params = [torch.zeros(len(g), dtype=torch.float64, requires_grad=True) for g in grads]
        for p, g in zip(params, grads):
            p.grad = torch.tensor(g, dtype=torch.float64)
        norm = float(torch.nn.utils.clip_grad_norm_(params, max_norm))
        flat = np.concatenate(grads).astype(np.float32)
        buckets = [(0, 100), (100, 37), (137, 1000)]
        s = GN.bucket_sumsq(flat, buckets, [1.0] * 3)
        assert np.isclose(GN.total_norm(s), norm, rtol=1e-6)
        coef = GN.clip_coef(GN.total_norm(s), max_norm)
        for p, (off, n) in zip(params, buckets):
            np.testing.assert_allclose(p.grad.numpy(), flat[off:off + n].astype(np.float64) * coef, rtol=1e-6,
                                       atol=1e-300)


def test_closed_forms():
    g = np.full(1000, 0.5, np.float32)
    s = GN.bucket_sumsq(g, [(0, 400), (400, 600)], [1.0, 0.25])
    assert s[0] == 400 * 0.25 and s[1] == 600 * (0.125 ** 2)
    assert GN.total_norm([9.0, 16.0]) == 5.0
    assert GN.clip_coef(5.0, 0.0) == 1.0 and GN.clip_coef(0.5, 1.0) == 1.0
    assert np.isclose(GN.clip_coef(10.0, 1.0), 1.0 / (10.0 + 1e-6))
    g[3] = np.nan
    g[500] = np.inf
    assert list(GN.bucket_nonfinite(g, [(0, 400), (400, 600)], [1.0, 1.0])) == [1, 1]


def test_factor_is_taken_in_fp32():
    g = np.ones(4, np.float32)
    assert GN.bucket_sumsq(g, [(0, 4)], [0.3])[0] == 4 * float(np.float32(0.3)) ** 2
