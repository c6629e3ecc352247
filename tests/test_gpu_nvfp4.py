"""Parity of the NVFP4 quantize kernels (bit-exact, with the tensor amax) and the NVFP4
forward GEMM (GPU), against the oracle of reading R16."""
import numpy as np
import pytest
import torch

import param_buffers_gb300 as gtp
from oracle import floats as F
from oracle import nvfp4 as NV
from param_buffers_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def quantize_gpu(x: torch.Tensor):
    R, C = x.shape
    p = torch.full((R, C // 2), 0xAB, dtype=torch.uint8, device=DEV)
    s = torch.full((R, C // 16), 0xAB, dtype=torch.uint8, device=DEV)
    a = torch.full((1,), 7.0, dtype=torch.float32, device=DEV)
    gtp.gtp_nvfp4_quantize_rowwise(x.to(DEV), p, s, a)
    torch.cuda.synchronize()
    return p, s, a


def adversarial(R, C, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((R, C)) * np.exp2(rng.integers(-12, 4, size=(R, 1)))).astype(np.float32)
    flat = x.reshape(-1, 16)
    n = flat.shape[0]
    flat[0] = 0.0                                                  # all-zero block
    if n > 8:
        flat[1, 7] = np.nan                                        # NaN block
        flat[2, 3] = -np.inf                                       # Inf block
        flat[3, :] = np.float32(2688.0)                            # the tensor amax: S = 1
        # S = 1 and amax_b = 6: sf = 1, so the elements themselves sit on E2M1 ties
        flat[4, :] = [6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 0.0, -0.0, 0.1, 5.9, 4.9, 1.0]
        flat[5, :] = 6.3                                           # sf rounds down: saturates at 6
        flat[5, 3] = -6.3
        flat[6, :] = np.float32(1e-40)                             # tiny block: zero scale
        flat[7, :] = -np.float32(2.0 ** -30)
    return x


@pytest.mark.parametrize("R,C", [(1, 16), (3, 48), (7, 160), (64, 2048), (1000, 272), (33, 4096)])
def test_quantize_fp32_bit_exact(R, C):
    x = adversarial(R, C, R * C)
    p, s, a = quantize_gpu(torch.from_numpy(x))
    rp, rs, ra = NV.quantize_rowwise(x)
    assert a.item() == float(ra)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(p.cpu().numpy(), rp)


@pytest.mark.parametrize("R,C", [(2, 32), (64, 2048), (1000, 272)])
def test_quantize_bf16_bit_exact(R, C):
    g = W.generator(R + C)
    x = W.randn_bf16((R, C), 1.0, g)
    p, s, a = quantize_gpu(x)
    rp, rs, ra = NV.quantize_rowwise(x.view(torch.int16).numpy().view(np.uint16), src_is_bf16_bits=True)
    assert a.item() == float(ra)
    assert np.array_equal(s.cpu().numpy(), rs) and np.array_equal(p.cpu().numpy(), rp)


def test_quantize_special_tensors():
    p, s, a = quantize_gpu(torch.zeros(4, 64))
    assert a.item() == 0.0 and not p.any().item() and not s.any().item()
    x = np.full((2, 32), np.float32(1e-40))                        # S clamps to FLT_MAX
    x[0, 0] = 0.0
    p, s, a = quantize_gpu(torch.from_numpy(x))
    rp, rs, _ = NV.quantize_rowwise(x)
    assert np.array_equal(p.cpu().numpy(), rp) and np.array_equal(s.cpu().numpy(), rs)
    e = torch.empty(0, 16)
    pe, se, ae = quantize_gpu(e)
    assert ae.item() == 0.0


def test_quantize_full_size_weights():
    """The MXFP8 workload's fp32 weights in NVFP4: W_fc1 [8192,2048], W_fc2 [2048,8192]."""
    g = W.generator(W.seed_of("mxfp8"))
    for name, R, C in W.MXFP8_W:
        x = W.randn_f32((R, C), 0.02, g)
        p, s, a = quantize_gpu(x)
        rp, rs, ra = NV.quantize_rowwise(x.numpy())
        assert a.item() == float(ra), name
        assert np.array_equal(s.cpu().numpy(), rs), name
        assert np.array_equal(p.cpu().numpy(), rp), name


def check_fprop(Yb, Xq, Xs, xa, Wq, Ws, wa, rows=None, cols=None):
    """rel. Frobenius <= 2e-3 against the float64 product of the dequantized operands, per
    element within one bf16 ulp plus the fp32 accumulation bound, >= 99% identical."""
    Xd, Wd = NV.dequantize_rowwise(Xq, Xs, xa), NV.dequantize_rowwise(Wq, Ws, wa)
    if rows is None:
        ref, absr = Xd @ Wd.T, np.abs(Xd) @ np.abs(Wd).T
    else:
        ref = np.einsum("ik,ik->i", Xd[rows], Wd[cols])
        absr = np.einsum("ik,ik->i", np.abs(Xd[rows]), np.abs(Wd[cols]))
    got = F.bf16_bits_to_f64(Yb)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 2e-3
    a = F.f64_to_bf16_bits(np.abs(ref))
    ulp = F.bf16_bits_to_f64(a + np.uint16(1)) - F.bf16_bits_to_f64(a)
    K = Xq.shape[1] * 2
    assert np.all(np.abs(got - ref) <= ulp + K * 2.0 ** -23 * absr + 4 * 2.0 ** -24 * np.abs(ref))
    assert (Yb == F.f64_to_bf16_bits(ref)).mean() >= 0.99


def run_fprop(X: torch.Tensor, Wt: torch.Tensor):
    M, K = X.shape
    N = Wt.shape[0]
    Xq, Xs, xa = (t for t in quantize_gpu(X))
    Wq, Ws, wa = (t for t in quantize_gpu(Wt))
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_fprop_nvfp4(Xq, Xs, xa, Wq, Ws, wa, Y)
    torch.cuda.synchronize()
    return Y.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.fixture(params=["single", "pair"])
def variant(request, monkeypatch):
    """Both block-scaled kernels: one CTA per tile, or a CTA pair per 256-row tile."""
    monkeypatch.setenv("GTP_GEMM_VARIANT", request.param)
    return request.param


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 512), (130, 264, 768), (1, 8, 256),
                                   (1000, 776, 1024), (512, 1024, 2048)])
def test_fprop_nvfp4(M, N, K, variant):
    g = W.generator(M + N + K + 5)
    X = W.randn_bf16((M, K), 1.0, g)
    Wt = W.randn_f32((N, K), 0.02, g)
    Yb = run_fprop(X, Wt)
    Xq, Xs, xa = NV.quantize_rowwise(X.view(torch.int16).numpy().view(np.uint16), src_is_bf16_bits=True)
    Wq, Ws, wa = NV.quantize_rowwise(Wt.numpy())
    check_fprop(Yb, Xq, Xs, xa, Wq, Ws, wa)


def test_fprop_nvfp4_full_size_sampled():
    """X bf16 [8192,2048] ~N(0,1) and W_fc1 fp32 [8192,2048] ~N(0,0.02), both in NVFP4."""
    g = W.generator(W.seed_of("mxfp8"))
    Wt = W.randn_f32(W.MXFP8_W[0][1:], 0.02, g)
    W.randn_f32(W.MXFP8_W[1][1:], 0.02, g)
    X = W.randn_bf16(W.MXFP8_X, 1.0, g)
    Yb = run_fprop(X, Wt)
    Xq, Xs, xa = NV.quantize_rowwise(X.view(torch.int16).numpy().view(np.uint16), src_is_bf16_bits=True)
    Wq, Ws, wa = NV.quantize_rowwise(Wt.numpy())
    rng = np.random.default_rng(6)
    r, c = rng.integers(0, 8192, 4096), rng.integers(0, 8192, 4096)
    check_fprop(Yb[r, c], Xq, Xs, xa, Wq, Ws, wa, r, c)
    last = np.full(8192, 8191)
    check_fprop(Yb[8191], Xq, Xs, xa, Wq, Ws, wa, last, np.arange(8192))


def test_nvfp4_errors():
    u = lambda *s: torch.zeros(*s, dtype=torch.uint8, device=DEV)
    a = torch.ones(1, device=DEV)
    with pytest.raises(gtp.GtpError, match="GTP_E_SHAPE"):
        gtp.gtp_linear_fprop_nvfp4(u(128, 64), u(128, 8), a, u(256, 64), u(256, 8), a,
                                   torch.empty(128, 256, dtype=torch.bfloat16, device=DEV))
    with pytest.raises(gtp.GtpError, match="GTP_E_SHAPE"):
        gtp.gtp_nvfp4_quantize_rowwise(torch.zeros(4, 24, device=DEV), u(4, 12), u(4, 1), a)
    Y = torch.full((128, 8), 1.0, dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_fprop_nvfp4(u(128, 0), u(128, 0), a, u(8, 0), u(8, 0), a, Y)   # K = 0: Y = 0
    torch.cuda.synchronize()
    assert not Y.any().item()
