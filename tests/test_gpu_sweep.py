"""Parity of the flat-buffer sweep kernels with the oracle (GPU).

Tolerances: AdamW state (master, m, v) relative Frobenius error <= 1e-6 against the
float64 oracle and per element |delta| <= 1e-6 * max|ref|; the bf16 param is the RNE
cast of the kernel's fp32 master bit for bit, and within one bf16 ulp of the cast of
the oracle's master; grad scaling and zeroing are bit-exact.
"""
import numpy as np
import pytest
import torch

import param_buffers_gb300 as gtp
from oracle import adamw as A
from oracle import floats as F
from param_buffers_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
H = A.AdamWHparams()
HP = gtp.AdamHparams(lr=H.lr, beta1=H.beta1, beta2=H.beta2, eps=H.eps, weight_decay=H.weight_decay)
RTOL_STATE = 1e-6


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def check_state(name, got: np.ndarray, ref: np.ndarray):
    got = got.astype(np.float64)
    nr = np.linalg.norm(ref)
    if nr == 0:
        assert not got.any(), name
        return
    rel = np.linalg.norm(got - ref) / nr
    assert rel <= RTOL_STATE, (name, rel)
    assert np.max(np.abs(got - ref)) <= RTOL_STATE * np.max(np.abs(ref)), name


def check_param(param_bits: np.ndarray, master_f32: np.ndarray, ref_master: np.ndarray):
    # bit-exact RNE of the kernel's own master (torch's cast on the CPU)
    own = torch.from_numpy(master_f32.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(param_bits, own)
    ref = F.f32_to_bf16_bits(ref_master.astype(np.float32))
    diff = np.abs(param_bits.astype(np.int64) - ref.astype(np.int64))
    assert diff.max() <= 1
    assert (diff != 0).mean() < 1e-3


def make_buckets(numel, rng, gaps=False):
    cuts = sorted(set(rng.integers(0, numel + 1, size=min(5, numel + 1)).tolist()) | {0, numel})
    out = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        if b <= a:
            continue
        if gaps and rng.random() < 0.3:
            continue
        out.append({"offset": a, "numel": b - a})
    # the C ABI takes fp32 factors: hand both sides the same fp32 value (0.3 is not exact)
    return out, [float(np.float32(rng.choice([0.5, 0.25, 1.0, 1 / 64, 0.3]))) for _ in out]


@pytest.mark.parametrize("numel", [1, 2, 3, 4, 5, 7, 1000, 4099, 131587, 1_000_003])
@pytest.mark.parametrize("gaps", [False, True])
def test_adam_step_small(numel, gaps):
    rng = np.random.default_rng(numel + gaps)
    g = W.generator(numel)
    grad, master, m, v, param = W.buffer_state(numel, g)
    # non-zero m, v so that later-step arithmetic is exercised too
    m.copy_(torch.randn(numel, generator=g) * 1e-4)
    v.copy_(torch.rand(numel, generator=g) * 1e-6)
    buckets, factors = make_buckets(numel, rng, gaps)
    fac = A.bucket_factor_per_element(numel, [(b["offset"], b["numel"]) for b in buckets], factors)
    ins = [t.numpy().copy() for t in (grad, master, m, v)]
    d = [t.to(DEV) for t in (grad, master, m, v, param)]
    gtp.gtp_adam_step_flat(*d, buckets, factors, HP, step=3)
    torch.cuda.synchronize()
    gs = A.scale_grad(ins[0], fac).astype(np.float64)
    P, M, V = A.adamw(ins[1], gs, ins[2], ins[3], 3, H)
    check_state("master", d[1].cpu().numpy(), P)
    check_state("exp_avg", d[2].cpu().numpy(), M)
    check_state("exp_avg_sq", d[3].cpu().numpy(), V)
    check_param(u16(d[4]), d[1].cpu().numpy(), P)
    assert torch.count_nonzero(d[0]).item() == 0


def test_adam_step_no_zero_and_empty():
    numel = 1029
    g = W.generator(5)
    grad, master, m, v, param = (t.to(DEV) for t in W.buffer_state(numel, g))
    g0 = grad.clone()
    gtp.gtp_adam_step_flat(grad, master, m, v, param, [], [], gtp.AdamHparams(zero_grad_after=False), step=1)
    torch.cuda.synchronize()
    assert torch.equal(grad, g0)
    e = torch.empty(0, device=DEV)
    gtp.gtp_adam_step_flat(e, e, e, e, torch.empty(0, dtype=torch.bfloat16, device=DEV), [], [], HP, step=1)


def test_cast_bit_exact_adversarial():
    """With lr = 0 the master is unchanged, so param_data must equal RNE_bf16(master) exactly."""
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    ties = ((rng.integers(0, 2 ** 16, size=50_000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000)
    x = np.concatenate([bits, ties]).view(np.float32)
    x = np.concatenate([x[np.isfinite(x)], np.array([np.finfo(np.float32).max, 3.3961e38, -0.0, 1e-45, 2.0 ** -134],
                                                    np.float32)])
    x = x[: (len(x) // 4) * 4 + 3]                      # ragged tail
    n = len(x)
    master = torch.from_numpy(x.copy()).to(DEV)
    grad = torch.zeros(n, device=DEV)
    m = torch.zeros(n, device=DEV)
    v = torch.zeros(n, device=DEV)
    param = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    gtp.gtp_adam_step_flat(grad, master, m, v, param, [], [],
                           gtp.AdamHparams(lr=0.0, weight_decay=0.0), step=1)
    torch.cuda.synchronize()
    assert np.array_equal(master.cpu().numpy().view(np.uint32), x.view(np.uint32))
    assert np.array_equal(u16(param), F.f32_to_bf16_bits(x))


def test_adam_three_steps():
    numel = 70_001
    g = W.generator(77)
    grad, master, m, v, param = W.buffer_state(numel, g)
    buckets = [{"offset": 0, "numel": 40_000}, {"offset": 40_000, "numel": numel - 40_000}]
    factors = [0.5, 0.25]
    fac = A.bucket_factor_per_element(numel, [(0, 40_000), (40_000, numel - 40_000)], factors)
    P, M, V = master.numpy().astype(np.float64), np.zeros(numel), np.zeros(numel)
    d = [t.to(DEV) for t in (grad, master, m, v, param)]
    for t in (1, 2, 3):
        gnew = W.randn_f32((numel,), 1e-3, g)
        d[0].copy_(gnew)
        gtp.gtp_adam_step_flat(*d, buckets, factors, HP, step=t)
        P, M, V = A.adamw(P, A.scale_grad(gnew.numpy(), fac).astype(np.float64), M, V, t, H)
    torch.cuda.synchronize()
    check_state("master", d[1].cpu().numpy(), P)
    check_state("exp_avg", d[2].cpu().numpy(), M)
    check_state("exp_avg_sq", d[3].cpu().numpy(), V)


def test_padding_stays_zero():
    """Reading R9: padding (zero grad/master/m/v) stays exactly zero through the sweep."""
    n = 4096
    d = [torch.zeros(n, device=DEV) for _ in range(4)] + [torch.full((n,), 7, dtype=torch.bfloat16, device=DEV)]
    gtp.gtp_adam_step_flat(*d, [{"offset": 0, "numel": n}], [0.5], HP, step=1)
    torch.cuda.synchronize()
    for t in d:
        assert torch.count_nonzero(t).item() == 0


def sampled_full_size(bw: W.BufferWorkload, n_samples: int):
    lay = gtp.gtp_buffer_layout([gtp.ParamDesc(p.numel, p.dtype, is_shared_embedding=p.is_shared_embedding)
                                 for p in bw.params],
                                gtp.LayoutConfig(bw.bucket_size, bw.dp_size, bw.use_distributed_optimizer,
                                                 bw.pad_buckets_for_high_nccl_busbw))
    numel = lay.buffers[0]["numel"]
    g = W.generator(W.seed_of(bw.name if bw.name != "7b" else "7b"), DEV)
    grad, master, m, v, param = W.buffer_state(numel, g, DEV, bw.grad_std, bw.param_std)
    pads = [(b["offset"] + b["numel_unpadded"], b["offset"] + b["numel"]) for b in lay.buckets]
    for a, z in pads:                       # the buffers are allocated zeroed: padding starts at 0
        for t in (grad, master, m, v, param):
            t[a:z].zero_()
    factors = [bw.gradient_scaling_factor] * len(lay.buckets)
    rng = np.random.default_rng(0)
    idx = rng.integers(0, numel, size=n_samples)
    edges = []
    for b in lay.buckets:
        for e in (b["offset"], b["offset"] + b["numel_unpadded"], b["offset"] + b["numel"]):
            edges += [e - 2, e - 1, e, e + 1]
    idx = np.unique(np.clip(np.concatenate([idx, np.array(edges), [0, numel - 1]]), 0, numel - 1))
    ti = torch.from_numpy(idx).to(DEV)
    ins = [t[ti].cpu().numpy() for t in (grad, master, m, v)]
    gtp.gtp_adam_step_flat(grad, master, m, v, param, lay.c_buckets, factors, HP, step=1)
    torch.cuda.synchronize()
    fac = np.ones(len(idx))
    for b, f in zip(lay.buckets, factors):
        fac[(idx >= b["offset"]) & (idx < b["offset"] + b["numel"])] = f
    gs = A.scale_grad(ins[0], fac).astype(np.float64)
    P, M, V = A.adamw(ins[1], gs, ins[2], ins[3], 1, H)
    check_state("master", master[ti].cpu().numpy(), P)
    check_state("exp_avg", m[ti].cpu().numpy(), M)
    check_state("exp_avg_sq", v[ti].cpu().numpy(), V)
    check_param(u16(param[ti]), master[ti].cpu().numpy(), P)
    assert torch.count_nonzero(grad).item() == 0
    # padding elements (if any) stay zero in every output
    for a, z in pads:
        for t in (master, m, v, param):
            assert torch.count_nonzero(t[a:z]).item() == 0


def test_stage_buffer_full_size_sampled():
    sampled_full_size(W.stage_buffer(), 1 << 20)


def test_7b_buffer_full_size_sampled():
    sampled_full_size(W.seven_b_buffer(), 1 << 20)


@pytest.mark.parametrize("numel", [1, 5, 4096, 100_003])
def test_bucket_scale_bit_exact_and_gaps_untouched(numel):
    rng = np.random.default_rng(numel)
    g = torch.randn(numel, generator=W.generator(numel)) * 1e-3
    buckets, factors = make_buckets(numel, rng, gaps=True)
    d = g.to(DEV)
    gtp.gtp_bucket_scale(d, buckets, factors)
    torch.cuda.synchronize()
    inb = np.zeros(numel, bool)
    fac = np.ones(numel)
    for b, f in zip(buckets, factors):
        inb[b["offset"]:b["offset"] + b["numel"]] = True
        fac[b["offset"]:b["offset"] + b["numel"]] = f
    want = np.where(inb, A.scale_grad(g.numpy(), fac), g.numpy())
    assert np.array_equal(d.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16, torch.uint8])
@pytest.mark.parametrize("numel", [1, 3, 16, 1000, 65_541])
def test_buffer_zero_with_guard_bands(dtype, numel):
    pad = 64 // torch.tensor([], dtype=dtype).element_size()        # keep the view 16-byte aligned
    base = torch.full((numel + 2 * pad,), 3, dtype=dtype, device=DEV)
    view = base[pad:pad + numel]
    gtp.gtp_buffer_zero(view)
    torch.cuda.synchronize()
    assert torch.count_nonzero(view).item() == 0
    assert torch.all(base[:pad] == 3).item() and torch.all(base[pad + numel:] == 3).item()


@pytest.mark.parametrize("numel", [1, 5, 4099, 131587, 1_000_003])
def test_adam_step_bf16_grad_buffer(numel):
    """A bf16 grad buffer (grad_reduce_in_fp32 off): the sweep converts each gradient to
    fp32 (step ① of the ZeRO-1 loop, exact for bf16) and otherwise runs the same AdamW,
    cast and zeroing; the oracle takes the same gradients as float64."""
    rng = np.random.default_rng(numel + 11)
    g = W.generator(numel + 11)
    _, master, m, v, param = W.buffer_state(numel, g)
    grad = W.randn_bf16((numel,), 1e-3, g)
    m.copy_(torch.randn(numel, generator=g) * 1e-4)
    v.copy_(torch.rand(numel, generator=g) * 1e-6)
    buckets, factors = make_buckets(numel, rng, gaps=True)
    fac = A.bucket_factor_per_element(numel, [(b["offset"], b["numel"]) for b in buckets], factors)
    ins = [grad.float().numpy().copy()] + [t.numpy().copy() for t in (master, m, v)]
    d = [t.to(DEV) for t in (grad, master, m, v, param)]
    gtp.gtp_adam_step_flat(*d, buckets, factors, HP, step=2)
    torch.cuda.synchronize()
    gs = A.scale_grad(ins[0], fac).astype(np.float64)
    P, M, V = A.adamw(ins[1], gs, ins[2], ins[3], 2, H)
    check_state("master", d[1].cpu().numpy(), P)
    check_state("exp_avg", d[2].cpu().numpy(), M)
    check_state("exp_avg_sq", d[3].cpu().numpy(), V)
    check_param(u16(d[4]), d[1].cpu().numpy(), P)
    assert d[0].dtype == torch.bfloat16 and torch.count_nonzero(d[0]).item() == 0
