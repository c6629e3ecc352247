"""The layer step's GEMMs at full size, in the launch configuration bench.py times (GPU).

One Llama-3.2-1B layer at TP=2 ("01 · ColumnParallelLinear / RowParallelLinear ...", §1
shard shapes), seq 8192, eight microbatches, in the overlap schedule: microbatch 0's
forward (four single launches), then for each microbatch its backward, linear by linear
in reverse, each linear's dgrad and wgrad accumulate grouped in one launch with the next
microbatch's forward of the linear at the same position of the forward chain; the last
microbatch's backward alone.  All wgrads accumulate into ONE flat fp32 grad_data at the
layout engine's offsets ("05 · grad/param buffer ...", §5, §6.2-§6.3).

Every launch writes its own outputs, so that all of them can be checked afterwards:
each Y and dX on 1024 sampled elements against the oracle's dot products (the bf16
GEMMs' bar: 2e-3 relative Frobenius, per element one bf16 ulp plus the fp32 accumulation
bound, 99 % rounded as the oracle rounds), and each main_grad view after the eight
microbatches on 2048 sampled elements against the oracle's per-call fp32 accumulate
(1e-5); the rest of grad_data stays +0.0.
"""
import numpy as np
import pytest
import torch

import param_buffers_gb300 as gtp
from oracle import gemm as G
from param_buffers_gb300 import workloads as W
from test_gpu_gemm import absbits, bits, check_bf16, rel

pytestmark = pytest.mark.gpu
DEV = "cuda"
WGRAD_TOL = 1e-5
NS = 1024


@pytest.fixture
def production_kernel(monkeypatch):
    for name in ("GTP_GEMM_VARIANT", "GTP_GEMM_SCHED", "GTP_GEMM_TAIL", "GTP_GEMM_L2HINT", "GTP_GROUP_SPLITS"):
        monkeypatch.delenv(name, raising=False)
    gtp.gtp_wait_timeouts(reset=True)
    yield
    assert gtp.gtp_wait_timeouts(reset=True) == 0


def test_overlap_schedule_full_size(production_kernel):
    bw = W.layer_buffer()
    lay = gtp.gtp_buffer_layout([gtp.ParamDesc(p.numel, p.dtype) for p in bw.params],
                                gtp.LayoutConfig(bw.bucket_size, bw.dp_size, True))
    numel = lay.buffers[0]["numel"]
    names = [p.name for p in bw.params]
    lins = W.LAYER_LINEARS
    off = {l.name: lay.index[names.index(l.name)]["start"] for l in lins}
    M, nmb = W.LAYER_M, W.LAYER_MICROBATCHES
    g = W.generator(W.seed_of("layer") + 123, DEV)
    Wt = {l.name: W.randn_bf16((l.N, l.K), 0.02, g, DEV) for l in lins}
    X = [{l.name: W.randn_bf16((M, l.K), 1.0, g, DEV) for l in lins} for _ in range(nmb)]
    dY = [{l.name: W.randn_bf16((M, l.N), 1.0, g, DEV) for l in lins} for _ in range(nmb)]
    Y = [{l.name: torch.empty(M, l.N, dtype=torch.bfloat16, device=DEV) for l in lins} for _ in range(nmb)]
    dX = [{l.name: torch.empty(M, l.K, dtype=torch.bfloat16, device=DEV) for l in lins} for _ in range(nmb)]
    grad = torch.full((numel,), float("nan"), device=DEV)
    gtp.gtp_buffer_zero(grad)

    # the schedule of bench.py's overlap step
    for l in lins:
        gtp.gtp_linear_fprop(X[0][l.name], Wt[l.name], Y[0][l.name])
    for mb in range(nmb):
        for lb, lf in zip(reversed(lins), lins):
            descs = [gtp.gemm_desc("dgrad", dY[mb][lb.name], Wt[lb.name], dX[mb][lb.name]),
                     gtp.gemm_desc("wgrad", dY[mb][lb.name], X[mb][lb.name], grad, off[lb.name])]
            if mb + 1 < nmb:
                descs.append(gtp.gemm_desc("fprop", X[mb + 1][lf.name], Wt[lf.name], Y[mb + 1][lf.name]))
            gtp.gtp_linear_grouped(descs)
    torch.cuda.synchronize()

    rng = np.random.default_rng(31)
    ar = np.arange(NS)
    for l in lins:
        n = l.name
        Wb = bits(Wt[n])
        for mb in range(nmb):
            r, c = rng.integers(0, M, NS), rng.integers(0, l.N, NS)        # Y [M, N]
            xr = bits(X[mb][n][torch.from_numpy(r).to(DEV)])
            got = bits(Y[mb][n][torch.from_numpy(r).to(DEV), torch.from_numpy(c).to(DEV)])
            check_bf16(got, G.sampled_fprop(xr, Wb[c], ar, ar), G.sampled_fprop(absbits(xr), absbits(Wb[c]), ar, ar),
                       l.K)
            r, c = rng.integers(0, M, NS), rng.integers(0, l.K, NS)        # dX [M, K]
            dyr = bits(dY[mb][n][torch.from_numpy(r).to(DEV)])
            got = bits(dX[mb][n][torch.from_numpy(r).to(DEV), torch.from_numpy(c).to(DEV)])
            check_bf16(got, G.sampled_dgrad(dyr, Wb[:, c], ar, ar),
                       G.sampled_dgrad(absbits(dyr), absbits(Wb[:, c]), ar, ar), l.N)
    out = grad.cpu().numpy()
    covered = np.zeros(numel, bool)
    for l in lins:
        n, o = l.name, off[l.name]
        rn, c = rng.integers(0, l.N, 2 * NS), rng.integers(0, l.K, 2 * NS)
        a2 = np.arange(2 * NS)
        ref = np.zeros(2 * NS, np.float32)
        for mb in range(nmb):
            dyc = bits(dY[mb][n][:, torch.from_numpy(rn).to(DEV)])
            xc = bits(X[mb][n][:, torch.from_numpy(c).to(DEV)])
            ref = G.sampled_wgrad_accum(ref, dyc, xc, a2, a2)
        view = out[o:o + l.N * l.K].reshape(l.N, l.K)
        assert rel(view[rn, c].astype(np.float64), ref.astype(np.float64)) <= WGRAD_TOL, n
        covered[o:o + l.N * l.K] = True
    rest = out[~covered]
    assert np.array_equal(rest.view(np.uint32), np.zeros(rest.size, np.uint32))
