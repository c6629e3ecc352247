"""Parity of the MXFP8 quantize kernel (bit-exact) and the MXFP8 fprop (GPU)."""
import numpy as np
import pytest
import torch

import param_buffers_gb300 as gtp
from oracle import floats as F
from oracle import gemm as G
from oracle import mxfp8 as MX
from param_buffers_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def quantize_gpu(x: torch.Tensor):
    R, C = x.shape
    q = torch.empty(R, C, dtype=torch.uint8, device=DEV)
    s = torch.empty(R, C // 32, dtype=torch.uint8, device=DEV)
    gtp.gtp_mxfp8_quantize_rowwise(x.to(DEV), q, s)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def adversarial(R, C, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((R, C)) * np.exp2(rng.integers(-40, 40, size=(R, 1)))
    x = x.astype(np.float32)
    flat = x.reshape(-1, 32)
    n = flat.shape[0]
    flat[0] = 0.0                                       # all-zero block
    if n > 3:
        flat[1, 7] = np.nan                             # NaN block
        flat[2, 3] = -np.inf                            # Inf block
        flat[3, :] = np.float32(1e-40)                  # subnormal amax
    if n > 8:
        flat[4, :] = 448.0 * 2.0 ** 5                   # exactly representable after scaling
        flat[5, 0] = np.float32(3.4e38)                 # near fp32 max
        flat[6, :] = -np.float32(2.0 ** -130)           # negative subnormals -> -0 codes
        # values on E4M3 rounding ties after scaling: amax 1.0 -> scale 2^-8 ... q = x * 256
        flat[7, :] = (np.arange(32) + 0.5) * 2.0 ** -8 * 8 / 32
        flat[8, :] = np.float32(465.0 / 256.0)          # rounds past 448 -> saturates
    return x


@pytest.mark.parametrize("R,C", [(1, 32), (3, 64), (7, 96), (64, 2048), (1000, 224)])
def test_quantize_fp32_bit_exact(R, C):
    x = adversarial(R, C, R * C)
    q, s = quantize_gpu(torch.from_numpy(x))
    rq, rs = MX.quantize_rowwise(x)
    assert np.array_equal(s, rs)
    assert np.array_equal(q, rq)


@pytest.mark.parametrize("R,C", [(2, 32), (129, 256), (4096, 2048)])
def test_quantize_bf16_bit_exact(R, C):
    x = W.randn_bf16((R, C), 1.0, W.generator(R + C))
    q, s = quantize_gpu(x)
    rq, rs = MX.quantize_rowwise(x.view(torch.int16).numpy().view(np.uint16), src_is_bf16_bits=True)
    assert np.array_equal(s, rs) and np.array_equal(q, rq)


def test_quantize_full_size_weights():
    """The FFN weights of the MXFP8 workload, fp32 master ~N(0, 0.02), bit-exact in full."""
    g = W.generator(W.seed_of("mxfp8"))
    for name, R, C in W.MXFP8_W:
        w = W.randn_f32((R, C), 0.02, g)
        q, s = quantize_gpu(w)
        rq, rs = MX.quantize_rowwise(w.numpy())
        assert np.array_equal(s, rs), name
        assert np.array_equal(q, rq), name


def check_fprop(Yb: np.ndarray, Xq, Xs, Wq, Ws, rows=None, cols=None):
    """rel. Frobenius <= 2e-3 against the float64 product of the dequantized operands, and
    per element within one bf16 ulp plus the fp32 accumulation bound K 2^-23 sum|terms|."""
    Xd, Wd = MX.dequantize_rowwise(Xq, Xs), MX.dequantize_rowwise(Wq, Ws)
    if rows is None:
        ref, absr = Xd @ Wd.T, np.abs(Xd) @ np.abs(Wd).T
    else:
        ref = np.einsum("ik,ik->i", Xd[rows], Wd[cols])
        absr = np.einsum("ik,ik->i", np.abs(Xd[rows]), np.abs(Wd[cols]))
    got = F.bf16_bits_to_f64(Yb)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 2e-3
    a = F.f64_to_bf16_bits(np.abs(ref))
    ulp = F.bf16_bits_to_f64(a + np.uint16(1)) - F.bf16_bits_to_f64(a)
    K = Xq.shape[1]
    assert np.all(np.abs(got - ref) <= ulp + K * 2.0 ** -23 * absr)
    assert (Yb == F.f64_to_bf16_bits(ref)).mean() >= 0.99


def run_fprop(X: torch.Tensor, Wt: torch.Tensor):
    """GPU path: quantize both operands on the GPU, then the block-scaled GEMM."""
    M, K = X.shape
    N = Wt.shape[0]
    Xq = torch.empty(M, K, dtype=torch.uint8, device=DEV)
    Xs = torch.empty(M, K // 32, dtype=torch.uint8, device=DEV)
    Wq = torch.empty(N, K, dtype=torch.uint8, device=DEV)
    Ws = torch.empty(N, K // 32, dtype=torch.uint8, device=DEV)
    gtp.gtp_mxfp8_quantize_rowwise(X.to(DEV), Xq, Xs)
    gtp.gtp_mxfp8_quantize_rowwise(Wt.to(DEV), Wq, Ws)
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_fprop_mxfp8(Xq, Xs, Wq, Ws, Y)
    torch.cuda.synchronize()
    return Y.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.fixture(params=["single", "pair"])
def variant(request, monkeypatch):
    """Both block-scaled kernels: one CTA per tile, or a CTA pair per 256-row tile."""
    monkeypatch.setenv("GTP_GEMM_VARIANT", request.param)
    return request.param


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 512, 256), (130, 264, 384), (1, 8, 128),
                                   (1000, 776, 1024), (512, 1024, 2048)])
def test_fprop_mxfp8(M, N, K, variant):
    g = W.generator(M + N + K)
    X = W.randn_bf16((M, K), 1.0, g)
    Wt = W.randn_f32((N, K), 0.02, g)
    Yb = run_fprop(X, Wt)
    Xq, Xs = MX.quantize_rowwise(X.view(torch.int16).numpy().view(np.uint16), src_is_bf16_bits=True)
    Wq, Ws = MX.quantize_rowwise(Wt.numpy())
    check_fprop(Yb, Xq, Xs, Wq, Ws)


@pytest.mark.parametrize("offset", [4, 2])
def test_fprop_mxfp8_unaligned_scale_views(offset, variant):
    """Scale views that start 4 (or 2) bytes into their storage, as a weight's view inside
    a native MXFP8 buffer does (scale offset = element offset / 32; parameters start on
    64-element boundaries): the CTA-pair kernel gathers such rows with loads instead of
    tensor copies.  2-byte alignment is refused (scales must be 4-byte aligned)."""
    M, N, K = 512, 768, 2048
    g = W.generator(M + N + K + offset)
    X = W.randn_bf16((M, K), 1.0, g)
    Wt = W.randn_f32((N, K), 0.02, g)
    Xq = torch.empty(M, K, dtype=torch.uint8, device=DEV)
    Wq = torch.empty(N, K, dtype=torch.uint8, device=DEV)
    xs_store = torch.empty(M * K // 32 + 64, dtype=torch.uint8, device=DEV)
    ws_store = torch.empty(N * K // 32 + 64, dtype=torch.uint8, device=DEV)
    Xs = xs_store[offset:offset + M * K // 32].view(M, K // 32)
    Ws = ws_store[offset:offset + N * K // 32].view(N, K // 32)
    gtp.gtp_mxfp8_quantize_rowwise(X.to(DEV), Xq, Xs)
    gtp.gtp_mxfp8_quantize_rowwise(Wt.to(DEV), Wq, Ws)
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    if offset % 4:
        with pytest.raises(gtp.GtpError):
            gtp.gtp_linear_fprop_mxfp8(Xq, Xs, Wq, Ws, Y)
        return
    gtp.gtp_linear_fprop_mxfp8(Xq, Xs, Wq, Ws, Y)
    torch.cuda.synchronize()
    Yb = Y.cpu().view(torch.int16).numpy().view(np.uint16)
    rXq, rXs = MX.quantize_rowwise(X.view(torch.int16).numpy().view(np.uint16), src_is_bf16_bits=True)
    rWq, rWs = MX.quantize_rowwise(Wt.numpy())
    check_fprop(Yb, rXq, rXs, rWq, rWs)


def test_fprop_mxfp8_full_size_sampled():
    """The MXFP8 workload: X bf16 [8192,2048] ~N(0,1), W_fc1 fp32 [8192,2048] ~N(0,0.02)."""
    g = W.generator(W.seed_of("mxfp8"))
    Wt = W.randn_f32(W.MXFP8_W[0][1:], 0.02, g)
    W.randn_f32(W.MXFP8_W[1][1:], 0.02, g)          # fc2 (drawn to keep the stream order)
    X = W.randn_bf16(W.MXFP8_X, 1.0, g)
    Yb = run_fprop(X, Wt)
    Xq, Xs = MX.quantize_rowwise(X.view(torch.int16).numpy().view(np.uint16), src_is_bf16_bits=True)
    Wq, Ws = MX.quantize_rowwise(Wt.numpy())
    rng = np.random.default_rng(5)
    r, c = rng.integers(0, 8192, 4096), rng.integers(0, 8192, 4096)
    check_fprop(Yb[r, c], Xq, Xs, Wq, Ws, r, c)
    last = np.full(8192, 8191)
    check_fprop(Yb[8191], Xq, Xs, Wq, Ws, last, np.arange(8192))


def quantize_col_gpu(x: torch.Tensor):
    R, C = x.shape
    q = torch.empty(C, R, dtype=torch.uint8, device=DEV)
    s = torch.empty(C, R // 32, dtype=torch.uint8, device=DEV)
    gtp.gtp_mxfp8_quantize_columnwise(x.to(DEV), q, s)
    torch.cuda.synchronize()
    return q, s


@pytest.mark.parametrize("R,C", [(32, 1), (64, 3), (96, 130), (160, 36), (224, 1028), (96, 128), (288, 264),
                                 (416, 520), (2048, 8192), (8192, 2048)])
def test_quantize_columnwise_bit_exact(R, C):
    x = adversarial(C, R, R + C).T.copy()          # special blocks land in columns
    q, s = quantize_col_gpu(torch.from_numpy(x))
    rq, rs = MX.quantize_columnwise(x)
    assert np.array_equal(s.cpu().numpy(), rs) and np.array_equal(q.cpu().numpy(), rq)
    xb = W.randn_bf16((R, C), 1.0, W.generator(R * C))
    q, s = quantize_col_gpu(xb)
    rq, rs = MX.quantize_columnwise(xb.view(torch.int16).numpy().view(np.uint16), src_is_bf16_bits=True)
    assert np.array_equal(s.cpu().numpy(), rs) and np.array_equal(q.cpu().numpy(), rq)


def test_quantize_columnwise_group_bit_exact():
    """Eight matrices in one call: fp32 and bf16 sources with NaN, Inf, zero, subnormal and
    saturating blocks in their columns, a ragged last column tile, an odd strip count, two
    matrices whose rows do not start on 16 bytes (cols 30 fp32, 36 bf16) and one whose
    source does not (a view at element 1), which take launches of their own, and an empty
    matrix.  Each view equals the oracle's columnwise quantization and the single call's."""
    shapes = [("f32", 256, 96), ("bf16", 128, 200), ("f32", 64, 30), ("bf16", 96, 36), ("f32", 0, 64),
              ("f32", 2048, 1028), ("bf16-offset", 64, 128), ("bf16", 160, 64)]
    views, refs = [], []
    for k, (kind, R, C) in enumerate(shapes):
        x = adversarial(C, R, 100 + k).T.copy() if R else np.zeros((0, C), np.float32)
        if kind == "f32":
            src = torch.from_numpy(x).to(DEV)
            refs.append(MX.quantize_columnwise(x) if R else None)
        else:
            xb = torch.from_numpy(x).to(torch.bfloat16)
            if kind == "bf16-offset":
                big = torch.empty(R * C + 1, dtype=torch.bfloat16, device=DEV)
                src = big[1:].view(R, C)
                src.copy_(xb)
            else:
                src = xb.to(DEV)
            refs.append(MX.quantize_columnwise(xb.view(torch.int16).numpy().view(np.uint16), src_is_bf16_bits=True))
        q = torch.full((C, R), 0xAB, dtype=torch.uint8, device=DEV)
        s = torch.full((C, R // 32), 0xCD, dtype=torch.uint8, device=DEV)
        views.append((src, q, s))
    gtp.gtp_mxfp8_quantize_columnwise_group(views)
    torch.cuda.synchronize()
    for (src, q, s), ref in zip(views, refs):
        if ref is None:
            continue
        assert np.array_equal(s.cpu().numpy(), ref[1]) and np.array_equal(q.cpu().numpy(), ref[0])
        q1, s1 = quantize_col_gpu(src)
        assert torch.equal(q1, q) and torch.equal(s1, s)


@pytest.mark.parametrize("R,C", [(96, 128), (160, 200), (2048, 8192)])
def test_quantize_columnwise_bf16_special_blocks(R, C):
    """bf16 sources with the special blocks (NaN, Inf, zero, subnormal, saturating) in their
    columns: the bf16 path keeps its column amax as packed 16-bit patterns."""
    x = adversarial(C, R, 7 * R + C).T.copy()
    xb = torch.from_numpy(x).to(torch.bfloat16)
    q, s = quantize_col_gpu(xb)
    rq, rs = MX.quantize_columnwise(xb.view(torch.int16).numpy().view(np.uint16), src_is_bf16_bits=True)
    assert np.array_equal(s.cpu().numpy(), rs) and np.array_equal(q.cpu().numpy(), rq)


def close_to(got: np.ndarray, ref: np.ndarray, absref: np.ndarray, K: int, bf16: bool):
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= (2e-3 if bf16 else 1e-5)
    if bf16:
        a = F.f64_to_bf16_bits(np.abs(ref))
        ulp = F.bf16_bits_to_f64(a + np.uint16(1)) - F.bf16_bits_to_f64(a)
    else:
        ulp = np.abs(ref) * 2.0 ** -23
    assert np.all(np.abs(got - ref) <= ulp + K * 2.0 ** -23 * absref)


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 384, 136), (1152, 640, 1032), (8192, 2048, 1024),
                                   (2560, 2048, 1024)])
def test_dgrad_and_wgrad_mxfp8(M, N, K, variant):
    """dX = dq(dY) dq(W^T)^T and main_grad += dq(dY^T) dq(X^T)^T on the columnwise views.

    (2560, 2048, 1024): the wgrad contraction of 20 stages splits in two, so the second
    unit starts at stage 10, inside a group of four stages whose scale bytes one tensor
    copy fetches on the CTA-pair kernel (scale rows of 80 bytes qualify for it)."""
    g = W.generator(M + 3 * N + 7 * K)
    X, Wt, dY = W.linear_inputs(M, N, K, g)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    # GPU path: quantize on the GPU, then the block-scaled GEMMs
    dYq = torch.empty(M, N, dtype=torch.uint8, device=DEV)
    dYs = torch.empty(M, N // 32, dtype=torch.uint8, device=DEV)
    gtp.gtp_mxfp8_quantize_rowwise(dY.to(DEV), dYq, dYs)
    Wtq, Wts = quantize_col_gpu(Wt)
    dX = torch.empty(M, K, dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_dgrad_mxfp8(dYq, dYs, Wtq, Wts, dX)
    dYtq, dYts = quantize_col_gpu(dY)
    Xtq, Xts = quantize_col_gpu(X)
    base = torch.randn(N * K + 8, generator=W.generator(5)) * 1e-3
    buf = base.to(DEV)
    gtp.gtp_linear_wgrad_accum_mxfp8(dYtq, dYts, Xtq, Xts, buf, 8)
    torch.cuda.synchronize()
    # oracle path: its own quantization of the same inputs
    rq, rs = MX.quantize_rowwise(bits(dY), src_is_bf16_bits=True)
    wq, ws = MX.quantize_columnwise(bits(Wt), src_is_bf16_bits=True)
    ref = MX.dgrad_mxfp8(rq, rs, wq, ws)
    absr = np.abs(MX.dequantize_rowwise(rq, rs)) @ np.abs(MX.dequantize_rowwise(wq, ws)).T
    close_to(F.bf16_bits_to_f64(dX.cpu().view(torch.int16).numpy().view(np.uint16)), ref, absr, N, True)
    dq, ds = MX.quantize_columnwise(bits(dY), src_is_bf16_bits=True)
    xq, xs = MX.quantize_columnwise(bits(X), src_is_bf16_bits=True)
    G0 = base.numpy()[8:].reshape(N, K)
    refw = MX.wgrad_accum_mxfp8(G0, dq, ds, xq, xs).astype(np.float64)
    absw = np.abs(G0) + np.abs(MX.dequantize_rowwise(dq, ds)) @ np.abs(MX.dequantize_rowwise(xq, xs)).T
    close_to(buf.cpu().numpy()[8:].reshape(N, K).astype(np.float64), refw, absw, M, False)
    assert np.array_equal(buf.cpu().numpy()[:8], base.numpy()[:8])


def test_quantize_errors():
    x = torch.zeros(4, 48, device=DEV)
    with pytest.raises((gtp.GtpError, ValueError)):
        gtp.gtp_mxfp8_quantize_rowwise(x, torch.empty(4, 48, dtype=torch.uint8, device=DEV),
                                       torch.empty(4, 1, dtype=torch.uint8, device=DEV))

