"""Parity of the native-MXFP8 optimizer sweep (gtp_adam_step_flat_mxfp8) with the oracle (GPU).

The fp32 state (master, m, v) follows the AdamW tolerances of the bf16 sweep; the MX
blocks are bit-exact against the oracle's quantization of the kernel's own fp32 master
(floating point decides the codes, so both sides decide from the same fp32 value), and
the master is bit-identical to the bf16 sweep's on the same inputs.
"""
import numpy as np
import pytest
import torch

import param_buffers_gb300 as gtp
from oracle import adamw as A
from oracle import mxfp8 as MX
from param_buffers_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
H = A.AdamWHparams()
HP = gtp.AdamHparams(lr=H.lr, beta1=H.beta1, beta2=H.beta2, eps=H.eps, weight_decay=H.weight_decay)
RTOL_STATE = 1e-6


def check_state(name, got: np.ndarray, ref: np.ndarray):
    got = got.astype(np.float64)
    nr = np.linalg.norm(ref)
    if nr == 0:
        assert not got.any(), name
        return
    assert np.linalg.norm(got - ref) / nr <= RTOL_STATE, name
    assert np.max(np.abs(got - ref)) <= RTOL_STATE * np.max(np.abs(ref)), name


def mx_outputs(n):
    return (torch.full((n,), 0xAB, dtype=torch.uint8, device=DEV),
            torch.full((n // 32,), 0xAB, dtype=torch.uint8, device=DEV))


@pytest.mark.parametrize("numel", [32, 4096, 131_072 + 7 * 32, 1_000_032])
@pytest.mark.parametrize("gaps", [False, True])
def test_mx_sweep_matches_oracle(numel, gaps):
    rng = np.random.default_rng(numel + 3 * gaps)
    g = W.generator(numel + 17)
    grad, master, m, v, param = W.buffer_state(numel, g)
    m.copy_(torch.randn(numel, generator=g) * 1e-4)
    v.copy_(torch.rand(numel, generator=g) * 1e-6)
    cuts = sorted(set(rng.integers(0, numel + 1, size=4).tolist()) | {0, numel})
    buckets = [{"offset": a, "numel": b - a} for a, b in zip(cuts[:-1], cuts[1:])
               if b > a and not (gaps and rng.random() < 0.3)]
    factors = [float(np.float32(rng.choice([0.5, 1 / 64, 0.3]))) for _ in buckets]
    fac = A.bucket_factor_per_element(numel, [(b["offset"], b["numel"]) for b in buckets], factors)
    ins = [t.numpy().copy() for t in (grad, master, m, v)]
    d = [t.to(DEV) for t in (grad, master, m, v)]
    ref = [t.to(DEV) for t in (grad, master, m, v, param)]
    q, s = mx_outputs(numel)
    gtp.gtp_adam_step_flat_mxfp8(*d, q, s, buckets, factors, HP, step=2)
    gtp.gtp_adam_step_flat(*ref, buckets, factors, HP, step=2)
    torch.cuda.synchronize()
    _, P, M, V, _, _ = A.fused_sweep_mxfp8(ins[0], ins[1], ins[2], ins[3], fac, 2, H)
    check_state("master", d[1].cpu().numpy(), P)
    check_state("exp_avg", d[2].cpu().numpy(), M)
    check_state("exp_avg_sq", d[3].cpu().numpy(), V)
    assert torch.count_nonzero(d[0]).item() == 0
    for a, b in zip(d[1:], ref[1:4]):                    # same arithmetic as the bf16 sweep
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    codes, scales = MX.quantize_flat_blocks(d[1].cpu().numpy())
    assert np.array_equal(q.cpu().numpy(), codes)
    assert np.array_equal(s.cpu().numpy(), scales)


def test_mx_sweep_special_blocks_bit_exact():
    """lr = 0 keeps the master: the blocks are the oracle's of the input itself, with NaN,
    Inf, all-zero, subnormal, saturating and tie values, and huge / tiny block scales."""
    rng = np.random.default_rng(5)
    n = 32 * 4096
    x = (rng.standard_normal(n) * np.exp2(rng.integers(-30, 30, size=n // 32).repeat(32))).astype(np.float32)
    x[0:32] = 0.0
    x[32 + 5] = np.nan
    x[64 + 31] = -np.inf
    x[96:128] = np.float32(1e-41)                                  # fp32 subnormals: scale byte 0
    x[128:160] = np.float32(3.0e38)
    x[160:192] = 1.0
    x[160] = 479.0                                                 # amax/scale in [448, 512): saturates
    x[192:224] = np.float32(1.0 + 1.0 / 16)                        # an E4M3 tie (between 1.0 and 1.125)
    x[192] = 1.0
    master = torch.from_numpy(x.copy()).to(DEV)
    z = [torch.zeros(n, device=DEV) for _ in range(3)]
    q, s = mx_outputs(n)
    gtp.gtp_adam_step_flat_mxfp8(z[0], master, z[1], z[2], q, s, [], [],
                                 gtp.AdamHparams(lr=0.0, weight_decay=0.0), step=1)
    torch.cuda.synchronize()
    got_master = master.cpu().numpy()
    assert np.array_equal(got_master.view(np.uint32)[np.isfinite(x)], x.view(np.uint32)[np.isfinite(x)])
    codes, scales = MX.quantize_flat_blocks(x)
    assert np.array_equal(q.cpu().numpy(), codes)
    assert np.array_equal(s.cpu().numpy(), scales)
    assert scales[0] == 0 and scales[1] == 0xFF and scales[2] == 0xFF and scales[3] == 0


def test_layer_weights_buffer_feeds_the_mxfp8_gemm():
    """The four weights of the layer as native MXFP8 parameters (storage dtype uint8, their
    own buffer) and the two norms in a bf16 buffer: after the sweep, each weight's slice of
    param_e4m3 / param_e8m0 equals the rowwise quantization of its master view, and the
    MXFP8 forward reading the slice directly equals the one reading a separate quantize."""
    shapes = {"qkv": (1536, 2048), "proj": (2048, 1024), "fc1": (8192, 2048), "fc2": (2048, 4096)}
    names = ["input_norm", "qkv", "proj", "mlp_norm", "fc1", "fc2"]
    descs = [gtp.ParamDesc(2048) if n.endswith("norm") else
             gtp.ParamDesc(shapes[n][0] * shapes[n][1], quantized_storage=True) for n in names]
    lay = gtp.gtp_buffer_layout(descs, gtp.LayoutConfig(40_000_000, 2))
    mx_buf = lay.index[names.index("fc1")]["buffer_id"]
    assert lay.index[names.index("input_norm")]["buffer_id"] != mx_buf
    numel = lay.buffers[mx_buf]["numel"]
    assert numel % 32 == 0
    bks = [b for b in lay.buckets if b["buffer_id"] == mx_buf]
    g = W.generator(W.seed_of("layer"), DEV)
    grad, master, m, v, _ = W.buffer_state(numel, g, DEV)
    q, s = mx_outputs(numel)
    gtp.gtp_adam_step_flat_mxfp8(grad, master, m, v, q, s, bks, [0.5] * len(bks), HP, step=1)
    X = W.randn_bf16((1024, 2048), 1.0, g, DEV)
    Xq = torch.empty(1024, 2048, dtype=torch.uint8, device=DEV)
    Xs = torch.empty(1024, 64, dtype=torch.uint8, device=DEV)
    gtp.gtp_mxfp8_quantize_rowwise(X, Xq, Xs)
    for n, (N, K) in shapes.items():
        st = lay.index[names.index(n)]["start"]
        assert lay.index[names.index(n)]["buffer_id"] == mx_buf and st % 32 == 0
        Wq, Ws = q[st:st + N * K].view(N, K), s[st // 32:(st + N * K) // 32].view(N, K // 32)
        rq = torch.empty(N, K, dtype=torch.uint8, device=DEV)
        rs = torch.empty(N, K // 32, dtype=torch.uint8, device=DEV)
        gtp.gtp_mxfp8_quantize_rowwise(master[st:st + N * K].view(N, K), rq, rs)
        torch.cuda.synchronize()
        assert torch.equal(Wq, rq) and torch.equal(Ws, rs), n
        if K == 2048:
            Y1 = torch.empty(1024, N, dtype=torch.bfloat16, device=DEV)
            Y2 = torch.empty_like(Y1)
            gtp.gtp_linear_fprop_mxfp8(Xq, Xs, Wq, Ws, Y1)
            gtp.gtp_linear_fprop_mxfp8(Xq, Xs, rq, rs, Y2)
            torch.cuda.synchronize()
            assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16)), n


def test_weight_at_a_128_element_offset():
    """A weight 128 elements into the buffer: its scale view starts 4 bytes in, which the
    GEMM accepts (4-byte scale loads); its codes start 128 bytes in."""
    N, K, M = 256, 512, 256
    g = W.generator(321, DEV)
    n = 128 + N * K + 128
    master = torch.zeros(n, device=DEV)
    master[128:128 + N * K] = W.randn_f32((N * K,), 0.02, g, DEV)
    z = [torch.zeros(n, device=DEV) for _ in range(3)]
    q, s = mx_outputs(n)
    gtp.gtp_adam_step_flat_mxfp8(z[0], master, z[1], z[2], q, s, [], [],
                                 gtp.AdamHparams(lr=0.0, weight_decay=0.0), step=1)
    Wq, Ws = q[128:128 + N * K].view(N, K), s[4:4 + N * K // 32].view(N, K // 32)
    rq = torch.empty(N, K, dtype=torch.uint8, device=DEV)
    rs = torch.empty(N, K // 32, dtype=torch.uint8, device=DEV)
    gtp.gtp_mxfp8_quantize_rowwise(master[128:128 + N * K].view(N, K), rq, rs)
    X = W.randn_bf16((M, K), 1.0, g, DEV)
    Xq = torch.empty(M, K, dtype=torch.uint8, device=DEV)
    Xs = torch.empty(M, K // 32, dtype=torch.uint8, device=DEV)
    gtp.gtp_mxfp8_quantize_rowwise(X, Xq, Xs)
    Y1 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    Y2 = torch.empty_like(Y1)
    gtp.gtp_linear_fprop_mxfp8(Xq, Xs, Wq, Ws, Y1)
    gtp.gtp_linear_fprop_mxfp8(Xq, Xs, rq, rs, Y2)
    torch.cuda.synchronize()
    assert torch.equal(Wq, rq) and torch.equal(Ws, rs)
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    assert Y1.abs().max().item() > 0
    with pytest.raises(gtp.GtpError, match="GTP_E_ALIGN"):
        gtp.gtp_linear_fprop_mxfp8(Xq, Xs, Wq, s[2:2 + N * K // 32].view(N, K // 32), Y1)


def test_mx_sweep_empty_and_shape_errors():
    e = torch.empty(0, device=DEV)
    u = torch.empty(0, dtype=torch.uint8, device=DEV)
    gtp.gtp_adam_step_flat_mxfp8(e, e, e, e, u, u, [], [], HP, step=1)
    n = 48
    d = [torch.zeros(n, device=DEV) for _ in range(4)]
    with pytest.raises(gtp.GtpError, match="GTP_E_SHAPE"):
        gtp.gtp_adam_step_flat_mxfp8(*d, torch.empty(n, dtype=torch.uint8, device=DEV),
                                     torch.empty(1, dtype=torch.uint8, device=DEV), [], [], HP, step=1)
