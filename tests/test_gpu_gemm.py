"""Parity of the tcgen05 GEMMs with the oracle (GPU).

Tolerance (stated for the GEMMs): relative Frobenius error <= 2e-3 against the float64
product of the same bf16 inputs.  Per element, a bf16 output is within one bf16 ulp of
the exact value plus the fp32 accumulation bound K * 2^-23 * sum_k |x_k w_k| (the
standard bound for a K-term fp32 sum, with a factor 2 for truncating adders); it
differs from the oracle's single RNE rounding only where that accumulation error
crosses a rounding boundary, which must be rare (>= 99% of elements identical).
wgrad accumulates into an fp32 view of a larger buffer whose guard bands must not change.
"""
import numpy as np
import pytest
import torch

import param_buffers_gb300 as gtp
from oracle import floats as F
from oracle import gemm as G
from param_buffers_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 2e-3


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def rel(a, b) -> float:
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb else float(np.linalg.norm(a))


def absbits(b: np.ndarray) -> np.ndarray:
    """|x| of bf16 bit patterns: the oracle applied to these gives sum_k |x_k w_k|."""
    return b & np.uint16(0x7FFF)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    a = F.f64_to_bf16_bits(np.abs(x))
    return F.bf16_bits_to_f64(a + np.uint16(1)) - F.bf16_bits_to_f64(a)


def check_bf16(got_bits: np.ndarray, ref64: np.ndarray, abs_sum: np.ndarray, K: int):
    got = F.bf16_bits_to_f64(got_bits)
    assert rel(got, ref64) <= TOL
    bound = bf16_ulp(ref64) + K * 2.0 ** -23 * abs_sum
    bad = np.abs(got - ref64) > bound
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], ref64[bad][:5])
    want = F.f64_to_bf16_bits(ref64)
    assert (got_bits == want).mean() >= 0.99


@pytest.fixture(params=["single", "pair-static", "pair-dynamic"])
def variant(request, monkeypatch):
    """Runs a test on the single-CTA kernel and on the CTA-pair kernel with both schedules."""
    kernel, _, sched = request.param.partition("-")
    monkeypatch.setenv("GTP_GEMM_VARIANT", kernel)
    monkeypatch.setenv("GTP_GEMM_SCHED", sched or "static")
    yield request.param
    assert gtp.gtp_wait_timeouts(reset=True) == 0


def inputs(M, N, K, seed):
    return W.linear_inputs(M, N, K, W.generator(seed))


SHAPES = [(1, 8, 8), (5, 16, 24), (128, 512, 256), (127, 264, 72), (130, 520, 200), (300, 256, 64),
          (257, 1000, 136), (64, 8, 1024), (513, 776, 584), (1024, 1536, 2048), (2000, 520, 1000)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_fprop_dgrad(M, N, K, variant):
    X, Wt, dY = inputs(M, N, K, M * 7 + N + K)
    dX_, dW_, ddY = X.to(DEV), Wt.to(DEV), dY.to(DEV)
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    dX = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_fprop(dX_, dW_, Y)
    gtp.gtp_linear_dgrad(ddY, dW_, dX)
    torch.cuda.synchronize()
    Xb, Wb, dYb = bits(X), bits(Wt), bits(dY)
    check_bf16(bits(Y), G.fprop(Xb, Wb), G.fprop(absbits(Xb), absbits(Wb)), K)
    check_bf16(bits(dX), G.dgrad(dYb, Wb), G.dgrad(absbits(dYb), absbits(Wb)), N)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_wgrad_accum_into_view(M, N, K, variant):
    X, Wt, dY = inputs(M, N, K, M + 3 * N + 5 * K)
    X2, _, dY2 = inputs(M, N, K, M + 3 * N + 5 * K + 1)
    guard = 64
    total = guard + N * K + guard
    base = torch.randn(total, generator=W.generator(N + K)) * 1e-3
    buf = base.to(DEV)
    gtp.gtp_linear_wgrad_accum(dY.to(DEV), X.to(DEV), buf, guard)
    gtp.gtp_linear_wgrad_accum(dY2.to(DEV), X2.to(DEV), buf, guard)
    torch.cuda.synchronize()
    out = buf.cpu().numpy()
    G0 = base.numpy()[guard:guard + N * K].reshape(N, K)
    ref = G.wgrad_accum(G.wgrad_accum(G0, bits(dY), bits(X)), bits(dY2), bits(X2))
    assert rel(out[guard:guard + N * K].reshape(N, K).astype(np.float64), ref.astype(np.float64)) <= TOL
    assert rel(out[guard:guard + N * K].reshape(N, K).astype(np.float64), ref.astype(np.float64)) <= 1e-5
    assert np.array_equal(out[:guard], base.numpy()[:guard])
    assert np.array_equal(out[guard + N * K:], base.numpy()[guard + N * K:])


def test_degenerate_shapes():
    Y = torch.full((4, 8), 3.0, dtype=torch.bfloat16, device=DEV)
    e = torch.empty(4, 0, dtype=torch.bfloat16, device=DEV)
    w0 = torch.empty(8, 0, dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_fprop(e, w0, Y)                    # K = 0: Y = 0
    dX = torch.full((4, 8), 3.0, dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_dgrad(torch.empty(4, 0, dtype=torch.bfloat16, device=DEV),
                         torch.empty(0, 8, dtype=torch.bfloat16, device=DEV), dX)   # N = 0: dX = 0
    g = torch.ones(64, device=DEV)
    gtp.gtp_linear_wgrad_accum(torch.empty(0, 8, dtype=torch.bfloat16, device=DEV),
                               torch.empty(0, 8, dtype=torch.bfloat16, device=DEV), g, 0)  # M = 0: no-op
    torch.cuda.synchronize()
    assert torch.count_nonzero(Y).item() == 0 and torch.count_nonzero(dX).item() == 0
    assert torch.all(g == 1).item()


def test_argument_errors():
    x = torch.zeros(16, 16, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(gtp.GtpError) as ei:
        gtp.gtp_linear_fprop(x, torch.zeros(12, 16, dtype=torch.bfloat16, device=DEV),
                             torch.zeros(16, 12, dtype=torch.bfloat16, device=DEV))
    assert "multiples of 8" in str(ei.value)
    g = torch.zeros(100, device=DEV)
    with pytest.raises(gtp.GtpError) as ei:
        gtp.gtp_linear_wgrad_accum(x, x, g, 0)        # 16*16 > 100
    assert "GTP_E_RANGE" in str(ei.value)


@pytest.mark.parametrize("lin", W.LAYER_LINEARS, ids=lambda l: l.name)
def test_layer_shapes_sampled(lin, variant):
    """Full Llama-3.2-1B TP=2 layer shapes (M = 8192): outputs checked on 4096 samples."""
    M, N, K = W.LAYER_M, lin.N, lin.K
    g = W.generator(W.seed_of("layer"), DEV)
    X, Wt, dY = W.linear_inputs(M, N, K, g, DEV)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    dX = torch.empty(M, K, dtype=torch.bfloat16, device=DEV)
    mg = torch.zeros(N * K + 64, device=DEV)
    gtp.gtp_linear_fprop(X, Wt, Y)
    gtp.gtp_linear_dgrad(dY, Wt, dX)
    gtp.gtp_linear_wgrad_accum(dY, X, mg, 64)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    Xb, Wb, dYb = bits(X), bits(Wt), bits(dY)
    r, c = rng.integers(0, M, 4096), rng.integers(0, N, 4096)
    check_bf16(bits(Y)[r, c], G.sampled_fprop(Xb, Wb, r, c), G.sampled_fprop(absbits(Xb), absbits(Wb), r, c), K)
    c2 = rng.integers(0, K, 4096)
    check_bf16(bits(dX)[r, c2], G.sampled_dgrad(dYb, Wb, r, c2), G.sampled_dgrad(absbits(dYb), absbits(Wb), r, c2), N)
    rn = rng.integers(0, N, 4096)
    got = mg[64:].view(N, K).cpu().numpy()[rn, c2].astype(np.float64)
    assert rel(got, G.sampled_wgrad(dYb, Xb, rn, c2)) <= 1e-5
    # corners and the last tile: full rows of the output against the oracle
    for i in (0, M - 1):
        rr, cc = np.full(N, i), np.arange(N)
        check_bf16(bits(Y)[i], G.sampled_fprop(Xb, Wb, rr, cc), G.sampled_fprop(absbits(Xb), absbits(Wb), rr, cc), K)
    assert torch.count_nonzero(mg[:64]).item() == 0


@pytest.mark.parametrize("lin", [l for l in W.LAYER_LINEARS if l.name in ("qkv", "fc1")], ids=lambda l: l.name)
def test_deterministic_wgrad_is_bit_reproducible(lin):
    """gtp_linear_wgrad_accum_deterministic: two identical sequences of three accumulating
    calls (the shapes the default entry point splits 3 and 2 ways) give bit-identical
    buffers, equal to the oracle's accumulate within the wgrad bar on 4096 samples."""
    M, N, K = W.LAYER_M, lin.N, lin.K
    g = W.generator(W.seed_of("layer") + 5, DEV)
    mbs = [(W.randn_bf16((M, K), 1.0, g, DEV), W.randn_bf16((M, N), 1.0, g, DEV)) for _ in range(3)]
    base = W.randn_f32((N * K + 128,), 1e-3, g, DEV)
    outs = []
    for _ in range(2):
        buf = base.clone()
        for X, dY in mbs:
            gtp.gtp_linear_wgrad_accum(dY, X, buf, 64, deterministic=True)
        outs.append(buf)
    torch.cuda.synchronize()
    a, b = (o.cpu().numpy().view(np.uint32) for o in outs)
    assert np.array_equal(a, b)
    rng = np.random.default_rng(3)
    r, c = rng.integers(0, N, 4096), rng.integers(0, K, 4096)
    ref = base[64:64 + N * K].view(N, K).cpu().numpy()[r, c]
    for X, dY in mbs:
        ref = G.sampled_wgrad_accum(ref, bits(dY), bits(X), r, c)
    got = outs[0][64:64 + N * K].view(N, K).cpu().numpy()[r, c].astype(np.float64)
    assert rel(got, ref.astype(np.float64)) <= 1e-5
    assert np.array_equal(a[:64], base[:64].cpu().numpy().view(np.uint32))
    assert np.array_equal(a[64 + N * K:], base[64 + N * K:].cpu().numpy().view(np.uint32))


# (300, 96, 64): 96 output rows, the single-CTA kernel's register epilogue
UNALIGNED = [(300, 256, 64), (513, 776, 584), (1024, 1536, 2048), (130, 264, 200), (300, 96, 64)]


@pytest.mark.parametrize("M,N,K", UNALIGNED)
@pytest.mark.parametrize("offset", [1, 2, 3, 6])
@pytest.mark.parametrize("deterministic", [False, True], ids=["split", "deterministic"])
def test_wgrad_into_unaligned_view(M, N, K, offset, deterministic):
    """A main_grad view at any element offset (the unpadded default layout), accumulated by
    fp32 atomic adds from registers: the oracle's per-call accumulate within the wgrad bar,
    the elements just before and after the view untouched."""
    X, _, dY = inputs(M, N, K, 31 * offset + M + N)
    X2, _, dY2 = inputs(M, N, K, 31 * offset + M + N + 1)
    total = offset + N * K + 37
    base = torch.randn(total, generator=W.generator(offset + K)) * 1e-3
    buf = base.to(DEV)
    for x, dy in ((X, dY), (X2, dY2)):
        gtp.gtp_linear_wgrad_accum(dy.to(DEV), x.to(DEV), buf, offset, deterministic=deterministic)
    torch.cuda.synchronize()
    out = buf.cpu().numpy()
    G0 = base.numpy()[offset:offset + N * K].reshape(N, K)
    ref = G.wgrad_accum(G.wgrad_accum(G0, bits(dY), bits(X)), bits(dY2), bits(X2))
    assert rel(out[offset:offset + N * K].reshape(N, K).astype(np.float64), ref.astype(np.float64)) <= 1e-5
    assert np.array_equal(out[:offset], base.numpy()[:offset])
    assert np.array_equal(out[offset + N * K:], base.numpy()[offset + N * K:])


def bf16_ulp_of_bits(b: np.ndarray) -> np.ndarray:
    a = b & np.uint16(0x7FFF)
    return F.bf16_bits_to_f64(a + np.uint16(1)) - F.bf16_bits_to_f64(a)


@pytest.mark.parametrize("M,N,K", [(300, 256, 64), (513, 776, 584), (1024, 1536, 2048), (64, 136, 72), (256, 120, 64)])
@pytest.mark.parametrize("offset", [0, 3, 64])
def test_wgrad_into_bf16_main_grad(M, N, K, offset):
    """A bf16 grad buffer (grad_reduce_in_fp32 off): two accumulating calls against the
    oracle's bf16 accumulate (one rounding of the exact sum a call).  The GPU rounds the fp32
    sum of its fp32 accumulator and the old value, so an element differs from the oracle
    only where fp32 accumulation error crosses a bf16 rounding boundary: at least 98 % are
    bit-identical, and each differs by at most one bf16 ulp of the first call's result
    (carried into the second) plus one of the second's, plus the fp32 accumulation bound
    M 2^-23 sum|dY X| of both calls; guard elements untouched; two runs bit-identical (no
    split contraction)."""
    X, _, dY = inputs(M, N, K, 7 * offset + M + 2 * N)
    X2, _, dY2 = inputs(M, N, K, 7 * offset + M + 2 * N + 1)
    total = offset + N * K + 24
    base = (torch.randn(total, generator=W.generator(offset + N)) * 4).to(torch.bfloat16)
    outs = []
    for _ in range(2):
        buf = base.to(DEV)
        for x, dy in ((X, dY), (X2, dY2)):
            gtp.gtp_linear_wgrad_accum(dy.to(DEV), x.to(DEV), buf, offset)
        outs.append(bits(buf))
    torch.cuda.synchronize()
    assert np.array_equal(outs[0], outs[1])
    out = outs[0]
    b0 = bits(base)
    ref1 = G.wgrad_accum_bf16(b0[offset:offset + N * K].reshape(N, K), bits(dY), bits(X))
    ref = G.wgrad_accum_bf16(ref1, bits(dY2), bits(X2))
    got = out[offset:offset + N * K].reshape(N, K)
    assert (got == ref).mean() >= 0.98
    diff = np.abs(F.bf16_bits_to_f64(got) - F.bf16_bits_to_f64(ref))
    acc = M * 2.0 ** -23 * (G.wgrad(absbits(bits(dY)), absbits(bits(X))) + G.wgrad(absbits(bits(dY2)), absbits(bits(X2))))
    bound = bf16_ulp_of_bits(ref1) + bf16_ulp_of_bits(ref) + acc
    assert np.all(diff <= bound), (diff - bound).max()
    assert np.array_equal(out[:offset], b0[:offset]) and np.array_equal(out[offset + N * K:], b0[offset + N * K:])
