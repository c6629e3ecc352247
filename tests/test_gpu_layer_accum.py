"""The layer workload's gradient accumulation at full size (GPU).

One Llama-3.2-1B layer at TP=2 ("01 · ColumnParallelLinear / RowParallelLinear ...",
§1 shard shapes): QKV [1536,2048], O [2048,1024], fc1 [8192,2048], fc2 [2048,4096], seq
8192.  Eight microbatches of all four wgrads accumulate into ONE flat fp32 grad_data at
the offsets the layout engine assigns ("05 · grad/param buffer ...", §5: main_grad is a
view of grad_data; §6.2-§6.3: gradients accumulate across microbatches under no_sync),
each call an in-place fp32 accumulate ([LIN] §4.2, gradient_accumulation_fusion).  The
library runs its production kernel here: the CTA pair, the static schedule and the
split counts it picks for each shape, so split partial tiles meet in main_grad through
fp32 reduce-adds on top of the eight per-call accumulations.

Checked against the oracle's sampled accumulate (one fp32 rounding per call, reading
R2) on 4096 random elements of each view plus one full row and one full column of it:
relative Frobenius error <= 1e-5 (the other wgrad tests' bar; the stated GEMM tolerance
is 2e-3).  Every element outside the four views (the two norms and padding) stays +0.0.
"""
import numpy as np
import pytest
import torch

import param_buffers_gb300 as gtp
from oracle import gemm as G
from param_buffers_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 2e-3
WGRAD_TOL = 1e-5


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def rel(a, b) -> float:
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.fixture
def production_kernel(monkeypatch):
    for name in ("GTP_GEMM_VARIANT", "GTP_GEMM_SCHED", "GTP_GEMM_TAIL", "GTP_GEMM_L2HINT"):
        monkeypatch.delenv(name, raising=False)
    gtp.gtp_wait_timeouts(reset=True)
    yield
    assert gtp.gtp_wait_timeouts(reset=True) == 0


def test_eight_microbatches_into_the_flat_buffer(production_kernel):
    bw = W.layer_buffer()
    lay = gtp.gtp_buffer_layout([gtp.ParamDesc(p.numel, p.dtype) for p in bw.params],
                                gtp.LayoutConfig(bw.bucket_size, bw.dp_size, True))
    numel = lay.buffers[0]["numel"]
    names = [p.name for p in bw.params]
    offsets = {lin.name: lay.index[names.index(lin.name)]["start"] for lin in W.LAYER_LINEARS}
    M = W.LAYER_M

    grad = torch.full((numel,), float("nan"), device=DEV)   # the iteration-start zero must clear it
    gtp.gtp_buffer_zero(grad)

    rng = np.random.default_rng(2024)
    groups = {}
    for lin in W.LAYER_LINEARS:
        n0, k0 = int(rng.integers(0, lin.N)), int(rng.integers(0, lin.K))
        groups[lin.name] = [
            (rng.integers(0, lin.N, 4096), rng.integers(0, lin.K, 4096)),        # random elements
            (np.full(lin.K, n0), np.arange(lin.K)),                             # one full row
            (np.arange(lin.N), np.full(lin.N, k0)),                             # one full column
        ]
    expect = {l.name: [np.zeros(len(r), np.float32) for r, _ in groups[l.name]] for l in W.LAYER_LINEARS}

    g = W.generator(W.seed_of("layer") + 99, DEV)
    for mb in range(W.LAYER_MICROBATCHES):
        for lin in W.LAYER_LINEARS:
            X = W.randn_bf16((M, lin.K), 1.0, g, DEV)
            dY = W.randn_bf16((M, lin.N), 1.0, g, DEV)
            gtp.gtp_linear_wgrad_accum(dY, X, grad, offsets[lin.name])
            Xb, dYb = bits(X), bits(dY)
            for i, (r, c) in enumerate(groups[lin.name]):
                expect[lin.name][i] = G.sampled_wgrad_accum(expect[lin.name][i], dYb, Xb, r, c)
    torch.cuda.synchronize()
    out = grad.cpu().numpy()

    covered = np.zeros(numel, bool)
    for lin in W.LAYER_LINEARS:
        o = offsets[lin.name]
        view = out[o:o + lin.N * lin.K].reshape(lin.N, lin.K)
        covered[o:o + lin.N * lin.K] = True
        for (r, c), ref in zip(groups[lin.name], expect[lin.name]):
            got = view[r, c].astype(np.float64)
            e = rel(got, ref.astype(np.float64))
            assert e <= TOL and e <= WGRAD_TOL, (lin.name, len(r), e)
    rest = out[~covered]
    assert rest.size == numel - sum(l.N * l.K for l in W.LAYER_LINEARS)
    assert np.array_equal(rest.view(np.uint32), np.zeros(rest.size, np.uint32))
