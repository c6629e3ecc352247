"""Grouped launches of the bf16 GEMMs (GPU): gtp_linear_backward (a linear's dgrad and
wgrad accumulate in one launch, "01 · ColumnParallelLinear / RowParallelLinear ...",
§4.2) and gtp_linear_grouped (up to four independent products in one launch).

Each product is held to the bar of its single entry point (the tests of test_gpu_gemm.py):
bf16 outputs within 2e-3 relative Frobenius error of the float64 product and per element
within one bf16 ulp plus the fp32 accumulation bound; main_grad views within 1e-5 of the
oracle's per-call fp32 accumulate, guard bands untouched.  Ragged shapes span several
tiles, a ragged last tile and the half-width tail; M <= 128 takes the single-CTA kernel
beside the group; wgrads into views the TMA cannot address (unaligned fp32, bf16 buffers)
take the register epilogues inside the group.  With GTP_GEMM_DETERMINISTIC two runs are
bit-identical.
"""
import numpy as np
import pytest
import torch

import param_buffers_gb300 as gtp
from oracle import floats as F
from oracle import gemm as G
from param_buffers_gb300 import workloads as W
from test_gpu_gemm import absbits, bf16_ulp_of_bits, bits, check_bf16, rel

pytestmark = pytest.mark.gpu
DEV = "cuda"
WGRAD_TOL = 1e-5


@pytest.fixture(autouse=True)
def clean_env(monkeypatch):
    for name in ("GTP_GEMM_VARIANT", "GTP_GEMM_SCHED", "GTP_GEMM_TAIL", "GTP_GROUP_SPLITS"):
        monkeypatch.delenv(name, raising=False)
    gtp.gtp_wait_timeouts(reset=True)
    yield
    assert gtp.gtp_wait_timeouts(reset=True) == 0


SHAPES = [(1, 8, 8), (128, 512, 256), (130, 520, 200), (300, 256, 64), (513, 776, 584), (1024, 1536, 2048),
          (2000, 520, 1000), (4096, 1024, 2048)]


def backward_case(M, N, K, seed, deterministic):
    X, Wt, dY = W.linear_inputs(M, N, K, W.generator(seed))
    X2, _, dY2 = W.linear_inputs(M, N, K, W.generator(seed + 1))
    guard = 64
    base = torch.randn(guard + N * K + guard, generator=W.generator(seed + 2)) * 1e-3
    buf = base.to(DEV)
    dX = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    dX2 = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    dW = Wt.to(DEV)
    gtp.gtp_linear_backward(dY.to(DEV), X.to(DEV), dW, dX, buf, guard, deterministic=deterministic)
    gtp.gtp_linear_backward(dY2.to(DEV), X2.to(DEV), dW, dX2, buf, guard, deterministic=deterministic)
    torch.cuda.synchronize()
    Wb = bits(Wt)
    for dy, dx in ((dY, dX), (dY2, dX2)):
        dyb = bits(dy)
        check_bf16(bits(dx), G.dgrad(dyb, Wb), G.dgrad(absbits(dyb), absbits(Wb)), N)
    out = buf.cpu().numpy()
    G0 = base.numpy()[guard:guard + N * K].reshape(N, K)
    ref = G.wgrad_accum(G.wgrad_accum(G0, bits(dY), bits(X)), bits(dY2), bits(X2))
    got = out[guard:guard + N * K].reshape(N, K).astype(np.float64)
    assert rel(got, ref.astype(np.float64)) <= WGRAD_TOL
    assert np.array_equal(out[:guard], base.numpy()[:guard])
    assert np.array_equal(out[guard + N * K:], base.numpy()[guard + N * K:])
    return out


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("deterministic", [False, True], ids=["split", "deterministic"])
def test_backward_matches_oracle(M, N, K, deterministic):
    backward_case(M, N, K, M + 7 * N + 11 * K, deterministic)


@pytest.mark.parametrize("M,N,K", [(2000, 520, 1000), (4096, 1024, 2048)])
def test_deterministic_backward_is_bit_reproducible(M, N, K):
    a = backward_case(M, N, K, 5, True)
    b = backward_case(M, N, K, 5, True)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("lin", W.LAYER_LINEARS, ids=lambda l: l.name)
def test_layer_backward_sampled(lin):
    """Full layer shapes (M = 8192): dX and the accumulated main_grad on 4096 samples plus a
    full row of dX, against the oracle."""
    M, N, K = W.LAYER_M, lin.N, lin.K
    g = W.generator(W.seed_of("layer") + 3, DEV)
    X, Wt, dY = W.linear_inputs(M, N, K, g, DEV)
    dX = torch.empty(M, K, dtype=torch.bfloat16, device=DEV)
    mg = torch.zeros(N * K + 64, device=DEV)
    gtp.gtp_linear_backward(dY, X, Wt, dX, mg, 64)
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    Xb, Wb, dYb = bits(X), bits(Wt), bits(dY)
    r, c = rng.integers(0, M, 4096), rng.integers(0, K, 4096)
    check_bf16(bits(dX)[r, c], G.sampled_dgrad(dYb, Wb, r, c), G.sampled_dgrad(absbits(dYb), absbits(Wb), r, c), N)
    i = M - 1
    rr, cc = np.full(K, i), np.arange(K)
    check_bf16(bits(dX)[i], G.sampled_dgrad(dYb, Wb, rr, cc), G.sampled_dgrad(absbits(dYb), absbits(Wb), rr, cc), N)
    rn = rng.integers(0, N, 4096)
    got = mg[64:].view(N, K).cpu().numpy()[rn, c].astype(np.float64)
    assert rel(got, G.sampled_wgrad(dYb, Xb, rn, c)) <= WGRAD_TOL
    assert torch.count_nonzero(mg[:64]).item() == 0


def test_grouped_four_mixed_products():
    """fprop, dgrad and two wgrads (into one buffer) of different shapes in one launch."""
    g = W.generator(606)
    X1, W1, _ = W.linear_inputs(640, 264, 136, g)          # fprop
    _, W2, dY2 = W.linear_inputs(1000, 512, 200, g)        # dgrad
    X3, _, dY3 = W.linear_inputs(2048, 768, 512, g)        # wgrad A
    X4, _, dY4 = W.linear_inputs(777, 392, 256, g)         # wgrad B (ragged M)
    off3, off4 = 128, 128 + 768 * 512 + 67                  # wgrad B's view is not 16-byte aligned
    total = off4 + 392 * 256 + 64
    base = torch.randn(total, generator=W.generator(607)) * 1e-3
    buf = base.to(DEV)
    Y1 = torch.full((640, 264), float("nan"), dtype=torch.bfloat16, device=DEV)
    dX2 = torch.full((1000, 200), float("nan"), dtype=torch.bfloat16, device=DEV)
    d = [t.to(DEV) for t in (X1, W1, W2, dY2, X3, dY3, X4, dY4)]
    descs = [gtp.gemm_desc("fprop", d[0], d[1], Y1), gtp.gemm_desc("dgrad", d[3], d[2], dX2),
             gtp.gemm_desc("wgrad", d[5], d[4], buf, off3), gtp.gemm_desc("wgrad", d[7], d[6], buf, off4)]
    gtp.gtp_linear_grouped(descs)
    torch.cuda.synchronize()
    check_bf16(bits(Y1), G.fprop(bits(X1), bits(W1)), G.fprop(absbits(bits(X1)), absbits(bits(W1))), 136)
    check_bf16(bits(dX2), G.dgrad(bits(dY2), bits(W2)), G.dgrad(absbits(bits(dY2)), absbits(bits(W2))), 512)
    out = buf.cpu().numpy()
    b0 = base.numpy()
    for off, (N, K), X, dY in ((off3, (768, 512), X3, dY3), (off4, (392, 256), X4, dY4)):
        ref = G.wgrad_accum(b0[off:off + N * K].reshape(N, K), bits(dY), bits(X))
        assert rel(out[off:off + N * K].reshape(N, K).astype(np.float64), ref.astype(np.float64)) <= WGRAD_TOL
    untouched = np.ones(total, bool)
    untouched[off3:off3 + 768 * 512] = False
    untouched[off4:off4 + 392 * 256] = False
    assert np.array_equal(out[untouched], b0[untouched])


def test_grouped_degenerate_and_small_products():
    """An empty contraction (zeros), an empty output (nothing) and an M <= 128 product
    (single-CTA kernel) beside a grouped one, in one call."""
    g = W.generator(808)
    Ye = torch.full((300, 64), 3.0, dtype=torch.bfloat16, device=DEV)
    Xs, Ws, _ = W.linear_inputs(100, 96, 48, g)
    Ys = torch.full((100, 96), float("nan"), dtype=torch.bfloat16, device=DEV)
    Xb_, Wb_, _ = W.linear_inputs(700, 304, 80, g)
    Yb = torch.full((700, 304), float("nan"), dtype=torch.bfloat16, device=DEV)
    descs = [gtp.gemm_desc("fprop", torch.empty(300, 0, dtype=torch.bfloat16, device=DEV),
                           torch.empty(64, 0, dtype=torch.bfloat16, device=DEV), Ye),
             gtp.gemm_desc("wgrad", torch.empty(0, 8, dtype=torch.bfloat16, device=DEV),
                           torch.empty(0, 8, dtype=torch.bfloat16, device=DEV), torch.ones(64, device=DEV)),
             gtp.gemm_desc("fprop", Xs.to(DEV), Ws.to(DEV), Ys),
             gtp.gemm_desc("fprop", Xb_.to(DEV), Wb_.to(DEV), Yb)]
    gtp.gtp_linear_grouped(descs)
    gtp.gtp_linear_grouped([])
    torch.cuda.synchronize()
    assert torch.count_nonzero(Ye).item() == 0
    for X, Wt, Y, K in ((Xs, Ws, Ys, 48), (Xb_, Wb_, Yb, 80)):
        check_bf16(bits(Y), G.fprop(bits(X), bits(Wt)), G.fprop(absbits(bits(X)), absbits(bits(Wt))), K)


def test_grouped_rejects_before_launching():
    x = torch.zeros(256, 64, dtype=torch.bfloat16, device=DEV)
    y = torch.full((256, 64), 7.0, dtype=torch.bfloat16, device=DEV)
    good = gtp.gemm_desc("fprop", x, torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV), y)
    bad = gtp.gemm_desc("wgrad", x, x, torch.zeros(100, device=DEV))       # 64*64 > 100: GTP_E_RANGE
    with pytest.raises(gtp.GtpError) as ei:
        gtp.gtp_linear_grouped([good, bad])
    assert "GTP_E_RANGE" in str(ei.value)
    torch.cuda.synchronize()
    assert torch.all(y == 7.0).item()                  # the valid product was not launched either


@pytest.mark.parametrize("deterministic", [False, True], ids=["split", "deterministic"])
def test_grouped_register_epilogues(deterministic):
    """Grouped wgrads that the TMA cannot write: two bf16 main_grad views (one at an odd
    element offset) and an fp32 view at an offset that is not 16-byte aligned, beside an
    fprop, in one launch, called twice.  The bf16 views are held to the bar of the single
    bf16 entry point (98 % bit-identical to the oracle's per-call bf16 accumulate, each
    element within the bf16 ulps of both calls' results plus the fp32 accumulation bound);
    the fp32 view to the per-call fp32 accumulate; guard elements untouched.  The bf16
    products are never split, so the bf16 buffer is bit-reproducible either way, and with
    GTP_GEMM_DETERMINISTIC so is the fp32 one."""
    g = W.generator(909)
    X1, W1, _ = W.linear_inputs(640, 264, 136, g)
    calls = [[W.linear_inputs(m, n, k, g) for m, n, k in ((1100, 392, 256), (513, 264, 200), (900, 520, 328))]
             for _ in range(2)]
    shapes = [(392, 256), (264, 200), (520, 328)]
    off_a, off_b, off_c = 16, 16 + 392 * 256 + 5, 67        # bf16 views a, b (odd); fp32 view c
    total_h, total_f = off_b + 264 * 200 + 24, off_c + 520 * 328 + 24
    base_h = (torch.randn(total_h, generator=W.generator(910)) * 4).to(torch.bfloat16)
    base_f = torch.randn(total_f, generator=W.generator(911)) * 1e-3
    runs = []
    for _ in range(2):
        bh, bf = base_h.to(DEV), base_f.to(DEV)
        Y1 = torch.full((640, 264), float("nan"), dtype=torch.bfloat16, device=DEV)
        for call in calls:
            (Xa, _, dYa), (Xb, _, dYb), (Xc, _, dYc) = [[t.to(DEV) for t in c] for c in call]
            gtp.gtp_linear_grouped([gtp.gemm_desc("fprop", X1.to(DEV), W1.to(DEV), Y1),
                                    gtp.gemm_desc("wgrad", dYa, Xa, bh, off_a),
                                    gtp.gemm_desc("wgrad", dYb, Xb, bh, off_b),
                                    gtp.gemm_desc("wgrad", dYc, Xc, bf, off_c)], deterministic=deterministic)
        torch.cuda.synchronize()
        runs.append((bits(bh), bf.cpu().numpy(), Y1))
    assert np.array_equal(runs[0][0], runs[1][0])
    if deterministic:
        assert np.array_equal(runs[0][1].view(np.uint32), runs[1][1].view(np.uint32))
    out_h, out_f, Y1 = runs[0]
    check_bf16(bits(Y1), G.fprop(bits(X1), bits(W1)), G.fprop(absbits(bits(X1)), absbits(bits(W1))), 136)
    b0 = bits(base_h)
    for j, off in ((0, off_a), (1, off_b)):
        N, K = shapes[j]
        (X, _, dY), (X2, _, dY2) = calls[0][j], calls[1][j]
        ref1 = G.wgrad_accum_bf16(b0[off:off + N * K].reshape(N, K), bits(dY), bits(X))
        ref = G.wgrad_accum_bf16(ref1, bits(dY2), bits(X2))
        got = out_h[off:off + N * K].reshape(N, K)
        assert (got == ref).mean() >= 0.98
        diff = np.abs(F.bf16_bits_to_f64(got) - F.bf16_bits_to_f64(ref))
        M = X.shape[0]
        acc = M * 2.0 ** -23 * (G.wgrad(absbits(bits(dY)), absbits(bits(X)))
                                + G.wgrad(absbits(bits(dY2)), absbits(bits(X2))))
        assert np.all(diff <= bf16_ulp_of_bits(ref1) + bf16_ulp_of_bits(ref) + acc)
    untouched = np.ones(total_h, bool)
    untouched[off_a:off_a + 392 * 256] = False
    untouched[off_b:off_b + 264 * 200] = False
    assert np.array_equal(out_h[untouched], b0[untouched])
    N, K = shapes[2]
    f0 = base_f.numpy()
    (X, _, dY), (X2, _, dY2) = calls[0][2], calls[1][2]
    ref = G.wgrad_accum(G.wgrad_accum(f0[off_c:off_c + N * K].reshape(N, K), bits(dY), bits(X)), bits(dY2), bits(X2))
    assert rel(out_f[off_c:off_c + N * K].reshape(N, K).astype(np.float64), ref.astype(np.float64)) <= WGRAD_TOL
    assert np.array_equal(out_f[:off_c], f0[:off_c]) and np.array_equal(out_f[off_c + N * K:], f0[off_c + N * K:])


def test_grouped_register_epilogues_small_outputs():
    """wgrads with at most 128 output rows (the single-CTA kernel, launched beside the group)
    into a bf16 buffer at an odd offset and an fp32 buffer at an offset that is not 16-byte
    aligned, next to a grouped fprop."""
    g = W.generator(913)
    Xa, _, dYa = W.linear_inputs(300, 96, 64, g)
    Xb, _, dYb = W.linear_inputs(257, 120, 64, g)
    X1, W1, _ = W.linear_inputs(384, 264, 72, g)
    off_a, off_b = 3, 5
    base_h = (torch.randn(off_a + 96 * 64 + 8, generator=W.generator(914)) * 4).to(torch.bfloat16)
    base_f = torch.randn(off_b + 120 * 64 + 8, generator=W.generator(915)) * 1e-3
    bh, bf = base_h.to(DEV), base_f.to(DEV)
    Y1 = torch.full((384, 264), float("nan"), dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_grouped([gtp.gemm_desc("wgrad", dYa.to(DEV), Xa.to(DEV), bh, off_a),
                            gtp.gemm_desc("wgrad", dYb.to(DEV), Xb.to(DEV), bf, off_b),
                            gtp.gemm_desc("fprop", X1.to(DEV), W1.to(DEV), Y1)])
    torch.cuda.synchronize()
    check_bf16(bits(Y1), G.fprop(bits(X1), bits(W1)), G.fprop(absbits(bits(X1)), absbits(bits(W1))), 72)
    b0 = bits(base_h)
    ref = G.wgrad_accum_bf16(b0[off_a:off_a + 96 * 64].reshape(96, 64), bits(dYa), bits(Xa))
    got = bits(bh)
    cur = got[off_a:off_a + 96 * 64].reshape(96, 64)
    assert (cur == ref).mean() >= 0.98
    diff = np.abs(F.bf16_bits_to_f64(cur) - F.bf16_bits_to_f64(ref))
    acc = 300 * 2.0 ** -23 * G.wgrad(absbits(bits(dYa)), absbits(bits(Xa)))
    assert np.all(diff <= bf16_ulp_of_bits(ref) + acc)
    assert np.array_equal(got[:off_a], b0[:off_a]) and np.array_equal(got[off_a + 96 * 64:], b0[off_a + 96 * 64:])
    f0 = base_f.numpy()
    out_f = bf.cpu().numpy()
    reff = G.wgrad_accum(f0[off_b:off_b + 120 * 64].reshape(120, 64), bits(dYb), bits(Xb))
    assert rel(out_f[off_b:off_b + 120 * 64].reshape(120, 64).astype(np.float64), reff.astype(np.float64)) <= WGRAD_TOL
    assert np.array_equal(out_f[:off_b], f0[:off_b]) and np.array_equal(out_f[off_b + 120 * 64:], f0[off_b + 120 * 64:])


@pytest.mark.parametrize("deterministic", [False, True], ids=["split", "deterministic"])
def test_grouped_two_microbatches_into_one_view(deterministic):
    """Two microbatches' wgrads of one linear into the same fp32 main_grad view in one launch
    (the group allows that overlap: fp32 additions commute): the oracle's accumulate of both
    calls within the wgrad bar, the elements around the view untouched."""
    g = W.generator(909)
    M, N, K = 2048, 768, 512
    X1, _, dY1 = W.linear_inputs(M, N, K, g)
    X2, _, dY2 = W.linear_inputs(M, N, K, g)
    off = 64
    total = off + N * K + 64
    base = torch.randn(total, generator=W.generator(910)) * 1e-3
    buf = base.to(DEV)
    d = [t.to(DEV) for t in (X1, dY1, X2, dY2)]
    gtp.gtp_linear_grouped([gtp.gemm_desc("wgrad", d[1], d[0], buf, off), gtp.gemm_desc("wgrad", d[3], d[2], buf, off)],
                           deterministic=deterministic)
    torch.cuda.synchronize()
    out, b0 = buf.cpu().numpy(), base.numpy()
    ref = G.wgrad_accum(G.wgrad_accum(b0[off:off + N * K].reshape(N, K), bits(dY1), bits(X1)), bits(dY2), bits(X2))
    assert rel(out[off:off + N * K].reshape(N, K).astype(np.float64), ref.astype(np.float64)) <= WGRAD_TOL
    assert np.array_equal(out[:off], b0[:off]) and np.array_equal(out[off + N * K:], b0[off + N * K:])


def test_grouped_rejects_overlapping_outputs():
    """A forward whose output overlaps another product's input is refused before launching:
    neither product runs."""
    x = torch.zeros(256, 64, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV)
    y = torch.full((256, 64), 7.0, dtype=torch.bfloat16, device=DEV)
    dy = torch.full((256, 64), 5.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(gtp.GtpError) as ei:
        gtp.gtp_linear_grouped([gtp.gemm_desc("fprop", x, w, y), gtp.gemm_desc("dgrad", y, w, dy)])   # reads y
    assert "GTP_E_ARG" in str(ei.value)
    torch.cuda.synchronize()
    assert torch.all(y == 7.0).item() and torch.all(dy == 5.0).item()
