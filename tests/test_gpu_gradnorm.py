"""Parity of the gradient-norm / non-finite / clip kernels with the oracle (GPU).

Per-bucket sums of squares, the total norm and the clip coefficient within 1e-6 relative
of the float64 oracle; non-finite counts exact; bit-identical results on repeated runs.
"""
import numpy as np
import pytest
import torch

import param_buffers_gb300 as gtp
from oracle import adamw as A
from oracle import gradnorm as GN
from param_buffers_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
RTOL = 1e-6


def buckets_for(numel, rng, gaps):
    cuts = sorted(set(rng.integers(0, numel + 1, size=min(6, numel + 1)).tolist()) | {0, numel})
    out = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        if b > a and not (gaps and rng.random() < 0.3):
            out.append({"offset": a, "numel": b - a})
    if not out:
        out = [{"offset": 0, "numel": numel}]
    factors = [float(np.float32(rng.choice([0.5, 1 / 64, 1.0, 0.3]))) for _ in out]
    return out, factors


def run_norm(grad: torch.Tensor, buckets, factors, max_norm):
    nb = len(buckets)
    ws = torch.empty(max(gtp.gtp_grad_norm_workspace_bytes(buckets), 16), dtype=torch.uint8, device=DEV)
    sumsq = torch.empty(nb, dtype=torch.float64, device=DEV)
    nonf = torch.empty(nb, dtype=torch.int32, device=DEV)
    tn = torch.empty(1, dtype=torch.float32, device=DEV)
    cc = torch.empty(1, dtype=torch.float32, device=DEV)
    gtp.gtp_grad_norm(grad, buckets, factors, max_norm, ws, sumsq, nonf, tn, cc)
    torch.cuda.synchronize()
    return sumsq.cpu().numpy(), nonf.cpu().numpy(), float(tn.item()), cc


def check(grad_np, buckets, factors, max_norm, got):
    spans = [(b["offset"], b["numel"]) for b in buckets]
    ref = GN.bucket_sumsq(grad_np, spans, factors)
    sumsq, nonf, tn, cc = got
    for s, r in zip(sumsq, ref):
        assert (s == 0 and r == 0) or abs(s - r) <= RTOL * r, (s, r)
    assert np.array_equal(nonf, GN.bucket_nonfinite(grad_np, spans, factors))
    norm = GN.total_norm(ref)
    assert abs(tn - norm) <= RTOL * norm + 1e-30
    assert abs(float(cc.item()) - GN.clip_coef(norm, max_norm)) <= RTOL * GN.clip_coef(norm, max_norm)


@pytest.mark.parametrize("numel", [1, 7, 4099, 131587, 1_000_003])
@pytest.mark.parametrize("gaps", [False, True])
def test_norm_small(numel, gaps):
    rng = np.random.default_rng(numel + gaps)
    g = W.randn_f32((numel,), 1e-3, W.generator(numel))
    buckets, factors = buckets_for(numel, rng, gaps)
    for max_norm in (0.0, 1.0, 1e-4):
        got = run_norm(g.to(DEV), buckets, factors, max_norm)
        check(g.numpy(), buckets, factors, max_norm, got)


def test_nonfinite_counts():
    n = 200_000
    g = W.randn_f32((n,), 1e-3, W.generator(3))
    g[17] = float("nan")
    g[150_001] = float("inf")
    g[150_002] = float("-inf")
    buckets = [{"offset": 0, "numel": 100_000}, {"offset": 100_000, "numel": 100_000}]
    sumsq, nonf, tn, cc = run_norm(g.to(DEV), buckets, [0.5, 0.5], 1.0)
    assert list(nonf) == [1, 2]
    assert not np.isfinite(tn)


def test_deterministic():
    g = W.randn_f32((3_000_017,), 1e-3, W.generator(9)).to(DEV)
    b = [{"offset": 0, "numel": 3_000_017}]
    a1 = run_norm(g, b, [0.25], 1.0)
    a2 = run_norm(g, b, [0.25], 1.0)
    assert a1[0].tobytes() == a2[0].tobytes() and a1[2] == a2[2]


def test_clip_feeds_the_sweep():
    """grad_norm's coefficient on the device drives the AdamW sweep (one fused step)."""
    n = 70_001
    g = W.generator(21)
    grad, master, m, v, param = W.buffer_state(n, g, grad_std=1.0)   # large gradients: clipping active
    buckets = [{"offset": 0, "numel": 40_000}, {"offset": 40_000, "numel": n - 40_000}]
    factors = [0.5, 0.5]
    ins = [t.numpy().copy() for t in (grad, master, m, v)]
    d = [t.to(DEV) for t in (grad, master, m, v, param)]
    sumsq, nonf, tn, cc = run_norm(d[0], buckets, factors, 1.0)
    gtp.gtp_adam_step_flat(*d, buckets, factors, gtp.AdamHparams(), step=1, grad_scale=cc)
    torch.cuda.synchronize()
    spans = [(b["offset"], b["numel"]) for b in buckets]
    coef = GN.clip_coef(GN.total_norm(GN.bucket_sumsq(ins[0], spans, factors)), 1.0)
    assert coef < 0.1
    fac = A.bucket_factor_per_element(n, spans, factors)
    gs = (A.scale_grad(ins[0], fac).astype(np.float64) * coef)
    P, M, V = A.adamw(ins[1], gs, ins[2], ins[3], 1, A.AdamWHparams())
    for got, ref in ((d[1], P), (d[2], M), (d[3], V)):
        x = got.cpu().numpy().astype(np.float64)
        assert np.linalg.norm(x - ref) <= 1e-6 * np.linalg.norm(ref)


def test_stage_buffer_full_size():
    bw = W.stage_buffer()
    lay = gtp.gtp_buffer_layout([gtp.ParamDesc(p.numel) for p in bw.params],
                                gtp.LayoutConfig(bw.bucket_size, bw.dp_size, True))
    numel = lay.buffers[0]["numel"]
    g = W.randn_f32((numel,), 1e-3, W.generator(W.seed_of("stage"), DEV), DEV)
    buckets = lay.buckets
    factors = [0.5] * len(buckets)
    got = run_norm(g, lay.c_buckets, factors, 1.0)
    check(g.cpu().numpy(), buckets, factors, 1.0, got)


def test_workspace_too_small():
    g = torch.zeros(1 << 20, device=DEV)
    b = [{"offset": 0, "numel": 1 << 20}]
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    out = [torch.empty(1, dtype=t, device=DEV) for t in (torch.float64, torch.int32, torch.float32, torch.float32)]
    with pytest.raises(gtp.GtpError) as ei:
        gtp.gtp_grad_norm(g, b, [1.0], 1.0, ws, *out)
    assert "GTP_E_CAPACITY" in str(ei.value)
