"""The tiled scale order on the GPU: the layout kernel and the tiled quantize outputs
against oracle/sf_layout.py, and the block-scaled GEMMs fed tiled scales against the same
GEMMs fed [rows, cols] scales (bit for bit) and against the float64 oracle product."""
import numpy as np
import pytest
import torch

import param_buffers_gb300 as gtp
from oracle import mxfp8 as MX
from oracle import nvfp4 as NV
from oracle import sf_layout as L
from param_buffers_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
FILL = 0xAB


def tiled_buffer(rows, cols):
    return torch.full((gtp.gtp_sf_tiled_bytes(rows, cols),), FILL, dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("rows,cols", [(1, 1), (5, 3), (128, 4), (130, 9), (1000, 64), (8192, 128), (257, 513)])
def test_sf_tile_matches_oracle(rows, cols):
    sf = np.random.default_rng(rows * 7 + cols).integers(0, 256, (rows, cols), dtype=np.uint8)
    out = tiled_buffer(rows, cols)
    gtp.gtp_sf_tile(torch.from_numpy(sf).to(DEV), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), L.tile_scales(sf))      # padding written as zero


@pytest.mark.parametrize("R,C", [(1, 32), (7, 96), (130, 288), (1000, 2048)])
def test_mxfp8_quantize_tiled(R, C):
    x = (np.random.default_rng(R + C).standard_normal((R, C)) * 0.02).astype(np.float32)
    q = torch.empty(R, C, dtype=torch.uint8, device=DEV)
    st = tiled_buffer(R, C // 32)
    gtp.gtp_mxfp8_quantize_rowwise_tiled(torch.from_numpy(x).to(DEV), q, st)
    torch.cuda.synchronize()
    rq, rs = MX.quantize_rowwise(x)
    assert np.array_equal(q.cpu().numpy(), rq)
    got = st.cpu().numpy()
    assert np.array_equal(L.untile_scales(got, R, C // 32), rs)
    pad = L.tile_scales(np.ones((R, C // 32), dtype=np.uint8)) == 0   # bytes that hold no scale
    assert np.all(got[pad] == FILL)                                    # left unwritten


@pytest.mark.parametrize("R,C", [(1, 16), (3, 48), (130, 272), (1000, 2048)])
def test_nvfp4_quantize_tiled(R, C):
    g = W.generator(R * 3 + C)
    x = W.randn_bf16((R, C), 1.0, g)
    p = torch.empty(R, C // 2, dtype=torch.uint8, device=DEV)
    st = tiled_buffer(R, C // 16)
    a = torch.full((1,), 7.0, dtype=torch.float32, device=DEV)
    gtp.gtp_nvfp4_quantize_rowwise_tiled(x.to(DEV), p, st, a)
    torch.cuda.synchronize()
    rp, rs, ra = NV.quantize_rowwise(x.view(torch.int16).numpy().view(np.uint16), src_is_bf16_bits=True)
    assert a.item() == float(ra)
    assert np.array_equal(p.cpu().numpy(), rp)
    got = st.cpu().numpy()
    assert np.array_equal(L.untile_scales(got, R, C // 16), rs)
    pad = L.tile_scales(np.ones((R, C // 16), dtype=np.uint8)) == 0
    assert np.all(got[pad] == FILL)


def tile_gpu(sf: torch.Tensor) -> torch.Tensor:
    out = tiled_buffer(*sf.shape)
    gtp.gtp_sf_tile(sf, out)
    return out


@pytest.fixture
def pair(monkeypatch):
    """The [rows, cols]-scale reference runs the same CTA-pair kernel as the tiled path."""
    monkeypatch.setenv("GTP_GEMM_VARIANT", "pair")


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 512), (130, 264, 768), (1, 8, 256),
                                   (1000, 776, 1024), (512, 1024, 2048)])
def test_fprop_nvfp4_tiled(M, N, K, pair):
    g = W.generator(M + N + K + 11)
    X = W.randn_bf16((M, K), 1.0, g)
    Wt = W.randn_f32((N, K), 0.02, g)
    q = lambda *s: torch.empty(*s, dtype=torch.uint8, device=DEV)
    Xq, Xs, Wq, Ws = q(M, K // 2), q(M, K // 16), q(N, K // 2), q(N, K // 16)
    xa, wa = torch.zeros(1, device=DEV), torch.zeros(1, device=DEV)
    gtp.gtp_nvfp4_quantize_rowwise(X.to(DEV), Xq, Xs, xa)
    gtp.gtp_nvfp4_quantize_rowwise(Wt.to(DEV), Wq, Ws, wa)
    Y0 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    Y1 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_fprop_nvfp4(Xq, Xs, xa, Wq, Ws, wa, Y0)
    gtp.gtp_linear_fprop_nvfp4_tiled(Xq, tile_gpu(Xs), xa, Wq, tile_gpu(Ws), wa, Y1)
    torch.cuda.synchronize()
    assert torch.equal(Y0.view(torch.int16), Y1.view(torch.int16))
    # and the oracle's product of the dequantized operands
    from test_gpu_nvfp4 import check_fprop
    Yb = Y1.cpu().view(torch.int16).numpy().view(np.uint16)
    rXq, rXs, rxa = NV.quantize_rowwise(X.view(torch.int16).numpy().view(np.uint16), src_is_bf16_bits=True)
    rWq, rWs, rwa = NV.quantize_rowwise(Wt.numpy())
    check_fprop(Yb, rXq, rXs, rxa, rWq, rWs, rwa)


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 512, 512), (130, 264, 384), (1, 8, 128),
                                   (1000, 776, 1024)])
def test_fprop_mxfp8_tiled(M, N, K, pair):
    g = W.generator(M + N + K + 13)
    X = W.randn_bf16((M, K), 1.0, g)
    Wt = W.randn_f32((N, K), 0.02, g)
    q = lambda *s: torch.empty(*s, dtype=torch.uint8, device=DEV)
    Xq, Xs, Wq, Ws = q(M, K), q(M, K // 32), q(N, K), q(N, K // 32)
    gtp.gtp_mxfp8_quantize_rowwise(X.to(DEV), Xq, Xs)
    gtp.gtp_mxfp8_quantize_rowwise(Wt.to(DEV), Wq, Ws)
    Y0 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    Y1 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_fprop_mxfp8(Xq, Xs, Wq, Ws, Y0)
    Xt, Wtl = tiled_buffer(M, K // 32), tiled_buffer(N, K // 32)
    gtp.gtp_mxfp8_quantize_rowwise_tiled(X.to(DEV), Xq, Xt)           # the fused tiled quantize
    gtp.gtp_mxfp8_quantize_rowwise_tiled(Wt.to(DEV), Wq, Wtl)
    gtp.gtp_linear_fprop_mxfp8_tiled(Xq, Xt, Wq, Wtl, Y1)
    torch.cuda.synchronize()
    assert torch.equal(Y0.view(torch.int16), Y1.view(torch.int16))


def test_fprop_nvfp4_tiled_full_size():
    """X bf16 [8192,2048] ~N(0,1) and W_fc1 fp32 [8192,2048] ~N(0,0.02): the tiled path
    (fused tiled quantize) equals the [rows, cols] path on every element."""
    g = W.generator(W.seed_of("mxfp8"))
    Wt = W.randn_f32(W.MXFP8_W[0][1:], 0.02, g)
    X = W.randn_bf16(W.MXFP8_X, 1.0, g)
    M, K = X.shape
    N = Wt.shape[0]
    q = lambda *s: torch.empty(*s, dtype=torch.uint8, device=DEV)
    Xq, Xs, Wq, Ws = q(M, K // 2), q(M, K // 16), q(N, K // 2), q(N, K // 16)
    xa, wa = torch.zeros(1, device=DEV), torch.zeros(1, device=DEV)
    Xd, Wd = X.to(DEV), Wt.to(DEV)
    gtp.gtp_nvfp4_quantize_rowwise(Xd, Xq, Xs, xa)
    gtp.gtp_nvfp4_quantize_rowwise(Wd, Wq, Ws, wa)
    Y0 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_fprop_nvfp4(Xq, Xs, xa, Wq, Ws, wa, Y0)
    Xt, Wtl = tiled_buffer(M, K // 16), tiled_buffer(N, K // 16)
    gtp.gtp_nvfp4_quantize_rowwise_tiled(Xd, Xq, Xt, xa)
    gtp.gtp_nvfp4_quantize_rowwise_tiled(Wd, Wq, Wtl, wa)
    Y1 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_fprop_nvfp4_tiled(Xq, Xt, xa, Wq, Wtl, wa, Y1)
    torch.cuda.synchronize()
    assert torch.equal(Y0.view(torch.int16), Y1.view(torch.int16))
    assert torch.isfinite(Y1.float()).all()


def test_tiled_errors():
    u = lambda *s: torch.zeros(*s, dtype=torch.uint8, device=DEV)
    a = torch.ones(1, device=DEV)
    Y = torch.empty(128, 256, dtype=torch.bfloat16, device=DEV)
    n = gtp.gtp_sf_tiled_bytes(128, 16)
    Xq, Wq, Wt = u(128, 128), u(256, 128), u(2 * n)
    with pytest.raises(ValueError):                                   # the tiled array's size is checked
        gtp.gtp_linear_fprop_nvfp4_tiled(Xq, u(n - 16), a, Wq, Wt, a, Y)
    buf = u(n + 16)                                                   # tiled scales must be 16-byte aligned
    st = gtp.lib().gtp_linear_fprop_nvfp4_tiled(Xq.data_ptr(), buf.data_ptr() + 4, a.data_ptr(), Wq.data_ptr(),
                                                Wt.data_ptr(), a.data_ptr(), Y.data_ptr(), 128, 256, 256,
                                                torch.cuda.current_stream().cuda_stream)
    assert st == gtp.abi.GTP_E_ALIGN
    with pytest.raises(gtp.GtpError, match="GTP_E_ALIGN"):
        gtp.gtp_sf_tile(u(4, 4), u(gtp.gtp_sf_tiled_bytes(4, 4) + 1)[1:])


@pytest.mark.parametrize("R,C", [(32, 8), (96, 130), (160, 264), (256, 36), (1024, 2048)])
def test_mxfp8_quantize_columnwise_tiled(R, C):
    """The columnwise view's scales in the tiled layout (rows = the source's columns): the
    oracle's [C, R/32] scales tiled, codes unchanged, padding left unwritten; fp32 and bf16
    sources (C = 130 and 36 take the strip kernel, the others the warp tiles)."""
    x = (np.random.default_rng(R * 5 + C).standard_normal((R, C)) * 0.02).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    for src, ref in ((torch.from_numpy(x), MX.quantize_columnwise(x)),
                     (xb, MX.quantize_columnwise(xb.view(torch.int16).numpy().view(np.uint16), src_is_bf16_bits=True))):
        q = torch.empty(C, R, dtype=torch.uint8, device=DEV)
        st = tiled_buffer(C, R // 32)
        gtp.gtp_mxfp8_quantize_columnwise_tiled(src.to(DEV), q, st)
        torch.cuda.synchronize()
        assert np.array_equal(q.cpu().numpy(), ref[0])
        got = st.cpu().numpy()
        assert np.array_equal(L.untile_scales(got, C, R // 32), ref[1])
        pad = L.tile_scales(np.ones((C, R // 32), dtype=np.uint8)) == 0
        assert np.all(got[pad] == FILL)


def test_mxfp8_quantize_columnwise_group_tiled():
    """A group mixing tiled and [C, R/32] scales: each view as its single call writes it."""
    rng = np.random.default_rng(41)
    srcs = [torch.from_numpy((rng.standard_normal((r, c)) * 0.02).astype(np.float32)).to(DEV)
            for r, c in ((256, 64), (96, 130), (128, 40))]
    srcs.append(torch.from_numpy(rng.standard_normal((160, 264)).astype(np.float32)).to(torch.bfloat16).to(DEV))
    views, refs = [], []
    for k, x in enumerate(srcs):
        R, C = x.shape
        q = torch.empty(C, R, dtype=torch.uint8, device=DEV)
        s = tiled_buffer(C, R // 32) if k % 2 == 0 else torch.empty(C, R // 32, dtype=torch.uint8, device=DEV)
        views.append((x, q, s))
        q1 = torch.empty_like(q)
        s1 = tiled_buffer(C, R // 32) if k % 2 == 0 else torch.empty_like(s)
        (gtp.gtp_mxfp8_quantize_columnwise_tiled if k % 2 == 0 else gtp.gtp_mxfp8_quantize_columnwise)(x, q1, s1)
        refs.append((q1, s1))
    gtp.gtp_mxfp8_quantize_columnwise_group(views)
    torch.cuda.synchronize()
    for (x, q, s), (q1, s1) in zip(views, refs):
        assert torch.equal(q, q1) and torch.equal(s, s1)


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (384, 512, 264), (1024, 1024, 776), (2048, 2048, 1024)])
def test_backward_mxfp8_tiled(M, N, K, pair):
    """MXFP8 dgrad and wgrad-accumulate fed tiled scales (the tiled quantize outputs) against
    the same GEMMs fed [rows, cols] scales on the CTA-pair kernel: dgrad bit for bit; the
    wgrad accumulate within the fp32 rounding of its split reduce-adds."""
    g = W.generator(M + 3 * N + K)
    X, Wt, dY = W.linear_inputs(M, N, K, g)
    Xd, Wd, dYd = X.to(DEV), Wt.to(DEV), dY.to(DEV)
    q = lambda *s: torch.empty(*s, dtype=torch.uint8, device=DEV)
    dYq, dYs, Wtq, Wts = q(M, N), q(M, N // 32), q(K, N), q(K, N // 32)
    dYtq, dYts, Xtq, Xts = q(N, M), q(N, M // 32), q(K, M), q(K, M // 32)
    gtp.gtp_mxfp8_quantize_rowwise(dYd, dYq, dYs)
    gtp.gtp_mxfp8_quantize_columnwise(Wd, Wtq, Wts)
    gtp.gtp_mxfp8_quantize_columnwise(dYd, dYtq, dYts)
    gtp.gtp_mxfp8_quantize_columnwise(Xd, Xtq, Xts)
    dYst, Wtst = tiled_buffer(M, N // 32), tiled_buffer(K, N // 32)
    dYtst, Xtst = tiled_buffer(N, M // 32), tiled_buffer(K, M // 32)
    gtp.gtp_mxfp8_quantize_rowwise_tiled(dYd, q(M, N), dYst)
    gtp.gtp_mxfp8_quantize_columnwise_group([(Wd, q(K, N), Wtst), (dYd, q(N, M), dYtst), (Xd, q(K, M), Xtst)])
    dX0 = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    dX1 = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_dgrad_mxfp8(dYq, dYs, Wtq, Wts, dX0)
    gtp.gtp_linear_dgrad_mxfp8_tiled(dYq, dYst, Wtq, Wtst, dX1)
    base = torch.randn(64 + N * K, generator=W.generator(M + N)) * 1e-3
    mg0, mg1 = base.to(DEV), base.to(DEV)
    gtp.gtp_linear_wgrad_accum_mxfp8(dYtq, dYts, Xtq, Xts, mg0, 64)
    gtp.gtp_linear_wgrad_accum_mxfp8_tiled(dYtq, dYtst, Xtq, Xtst, mg1, 64)
    torch.cuda.synchronize()
    assert torch.equal(dX0.view(torch.int16), dX1.view(torch.int16))
    a, b = mg0.cpu().double(), mg1.cpu().double()
    assert torch.equal(a[:64], base[:64].double())
    assert (a - b).norm() <= 1e-6 * a.norm()
    assert torch.all((a - b).abs() <= 8 * 2.0 ** -23 * a.abs().max())


def test_mxfp8_quantize_rowwise_group():
    """fp32 and bf16 matrices, [R, C/32] and tiled scales, an empty one, in one launch:
    each as its single call writes it, and the oracle's codes and scales (NaN, Inf, zero
    and subnormal blocks included)."""
    rng = np.random.default_rng(77)
    shapes = [("f32", 130, 288, False), ("bf16", 64, 2048, True), ("f32", 0, 64, False),
              ("f32", 1000, 224, True), ("bf16", 7, 96, False)]
    views, refs = [], []
    for kind, R, C, tiled in shapes:
        from test_gpu_mxfp8 import adversarial
        x = adversarial(R, C, R + C) if R else np.zeros((0, C), np.float32)
        if kind == "f32":
            src = torch.from_numpy(x).to(DEV)
            ref = MX.quantize_rowwise(x) if R else None
        else:
            xb = torch.from_numpy(x).to(torch.bfloat16)
            src = xb.to(DEV)
            ref = MX.quantize_rowwise(xb.view(torch.int16).numpy().view(np.uint16), src_is_bf16_bits=True)
        q = torch.full((R, C), 0xAB, dtype=torch.uint8, device=DEV)
        s = tiled_buffer(R, C // 32) if tiled else torch.full((R, C // 32), 0xCD, dtype=torch.uint8, device=DEV)
        views.append((src, q, s))
        refs.append((ref, tiled, R, C))
    gtp.gtp_mxfp8_quantize_rowwise_group(views)
    torch.cuda.synchronize()
    for (src, q, s), (ref, tiled, R, C) in zip(views, refs):
        if ref is None:
            continue
        assert np.array_equal(q.cpu().numpy(), ref[0])
        got = s.cpu().numpy()
        assert np.array_equal(L.untile_scales(got, R, C // 32) if tiled else got, ref[1])
        q1, s1 = torch.empty_like(q), torch.empty_like(s)
        (gtp.gtp_mxfp8_quantize_rowwise_tiled if tiled else gtp.gtp_mxfp8_quantize_rowwise)(src, q1, s1)
        torch.cuda.synchronize()
        assert torch.equal(q1, q)


def test_step_mxfp8_part_full_size(pair):
    """The layer step's MXFP8 part at full size, as bench.py launches it: the fc1 and fc2
    fp32 masters and fc1's bf16 input quantized rowwise by one grouped call with tiled
    scales, then the tiled MXFP8 fc1 forward -- equal to separate [rows, cols]-scale
    quantizes (codes bit for bit, scales untiled) and to the [rows, cols]-scale forward on
    the same CTA-pair kernel, bit for bit."""
    g = W.generator(W.seed_of("mxfp8") + 5, DEV)
    W1 = W.randn_f32((8192, 2048), 0.02, g, DEV)
    W2 = W.randn_f32((2048, 8192), 0.02, g, DEV)
    X = W.randn_bf16((8192, 2048), 1.0, g, DEV)
    q = lambda *s: torch.empty(*s, dtype=torch.uint8, device=DEV)
    outs = [(q(*t.shape), tiled_buffer(t.shape[0], t.shape[1] // 32)) for t in (W1, W2, X)]
    gtp.gtp_mxfp8_quantize_rowwise_group([(t, a, b) for t, (a, b) in zip((W1, W2, X), outs)])
    Y1 = torch.empty(8192, 8192, dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_fprop_mxfp8_tiled(outs[2][0], outs[2][1], outs[0][0], outs[0][1], Y1)
    ref = [(q(*t.shape), q(t.shape[0], t.shape[1] // 32)) for t in (W1, W2, X)]
    for t, (a, b) in zip((W1, W2, X), ref):
        gtp.gtp_mxfp8_quantize_rowwise(t, a, b)
    Y0 = torch.empty(8192, 8192, dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_fprop_mxfp8(ref[2][0], ref[2][1], ref[0][0], ref[0][1], Y0)
    torch.cuda.synchronize()
    for t, (a, b), (ra, rb) in zip((W1, W2, X), outs, ref):
        assert torch.equal(a, ra)
        assert np.array_equal(L.untile_scales(b.cpu().numpy(), t.shape[0], t.shape[1] // 32), rb.cpu().numpy())
    assert torch.equal(Y0.view(torch.int16), Y1.view(torch.int16))
