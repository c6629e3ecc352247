"""Pins of the optimizer-sweep oracle: torch's AdamW in float64, the t=1 closed form,
the scalar loop, padding invariance and sharding invariance."""
import numpy as np
import pytest
import torch

from oracle import adamw as A
from oracle import floats as F

H = A.AdamWHparams()


def state(n, seed=0, nonzero_mv=False):
    rng = np.random.default_rng(seed)
    p = rng.standard_normal(n) * 0.02
    g = rng.standard_normal(n) * 1e-3
    m = rng.standard_normal(n) * 1e-4 if nonzero_mv else np.zeros(n)
    v = rng.random(n) * 1e-6 if nonzero_mv else np.zeros(n)
    return p, g, m, v


@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_matches_torch_adamw_float64(wd):
    """torch.optim.AdamW (single-tensor path, float64) over three steps."""
    h = A.AdamWHparams(weight_decay=wd)
    p0, _, _, _ = state(1000, 1)
    P = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([P], lr=h.lr, betas=(h.beta1, h.beta2), eps=h.eps, weight_decay=h.weight_decay,
                            foreach=False)
    p, m, v = p0.copy(), np.zeros(1000), np.zeros(1000)
    rng = np.random.default_rng(7)
    for t in (1, 2, 3):
        g = rng.standard_normal(1000) * 1e-3
        P.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        p, m, v = A.adamw(p, g, m, v, t, h)
        st = opt.state[P]
        np.testing.assert_allclose(P.detach().numpy(), p, rtol=1e-13, atol=1e-17)
        np.testing.assert_allclose(st["exp_avg"].numpy(), m, rtol=1e-13, atol=1e-20)
        np.testing.assert_allclose(st["exp_avg_sq"].numpy(), v, rtol=1e-13, atol=1e-25)


def test_first_step_closed_form():
    """t=1 from m=v=0: m_hat = g, v_hat = g^2, so p <- p(1 - lr wd) - lr g / (|g| + eps)."""
    p, g, m, v = state(5000, 2)
    P, M, V = A.adamw(p, g, m, v, 1, H)
    np.testing.assert_allclose(P, p * (1 - H.lr * H.weight_decay) - H.lr * g / (np.abs(g) + H.eps), rtol=1e-12)
    np.testing.assert_allclose(M, (1 - H.beta1) * g, rtol=1e-15)
    np.testing.assert_allclose(V, (1 - H.beta2) * g * g, rtol=1e-15)


def test_scalar_loop_equals_vector_form():
    p, g, m, v = state(300, 3, nonzero_mv=True)
    a = A.adamw_loop(p, g, m, v, 5, H)
    b = A.adamw(p, g, m, v, 5, H)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-15, atol=0)


def test_padding_stays_zero():
    """Reading R9: zero grad, master, m, v stay exactly zero through the update."""
    z = np.zeros(10)
    P, M, V = A.adamw(z, z, z, z, 1, H)
    assert not P.any() and not M.any() and not V.any()
    _, p, m, v, prm = A.fused_sweep(z.astype(np.float32), z, z, z, np.ones(10), 1, H)
    assert not p.any() and not prm.any()


def test_sharding_invariance():
    """[MLM] §6.4 toy: dp-sharded Adam equals single-process Adam (elementwise, so exactly)."""
    p, g, m, v = state(22, 4, nonzero_mv=True)
    whole = A.adamw(p, g, m, v, 2, H)
    parts = [A.adamw(p[a:b], g[a:b], m[a:b], v[a:b], 2, H) for a, b in ((0, 11), (11, 22))]
    for k in range(3):
        assert np.array_equal(np.concatenate([parts[0][k], parts[1][k]]), whole[k])


def test_fused_sweep_composition():
    """scale -> AdamW -> bf16 cast -> zero, with one factor per bucket."""
    n = 1000
    rng = np.random.default_rng(5)
    grad = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    master = (rng.standard_normal(n) * 0.02).astype(np.float32)
    buckets = [(0, 400), (400, 600)]
    factors = [0.5, 0.25]
    fac = A.bucket_factor_per_element(n, buckets, factors)
    assert fac[0] == 0.5 and fac[399] == 0.5 and fac[400] == 0.25 and fac[-1] == 0.25
    g_out, p, m, v, prm = A.fused_sweep(grad, master, np.zeros(n), np.zeros(n), fac, 1, H)
    assert not g_out.any()
    gs = grad.astype(np.float64) * fac            # powers of two: exact
    np.testing.assert_array_equal(A.scale_grad(grad, fac).astype(np.float64), gs)
    P, M, V = A.adamw(master, gs, np.zeros(n), np.zeros(n), 1, H)
    np.testing.assert_array_equal(p, P)
    assert np.array_equal(prm, torch.from_numpy(P.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(prm, F.f32_to_bf16_bits(P.astype(np.float32)))
