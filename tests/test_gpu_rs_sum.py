"""The local fp32 sum of the all-to-all reduce-scatter on the GPU ([BUF] §9.1) against
oracle/rs_sum.py: bit for bit, since both add the slices in rank order with one fp32
rounding per addition and round once to a bf16 output."""
import numpy as np
import pytest
import torch

import param_buffers_gb300 as gtp
from oracle import floats as F
from oracle import rs_sum as R
from param_buffers_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def slices_of(P, n, in_bf16, seed):
    g = torch.Generator().manual_seed(seed)
    scale = torch.exp2(torch.randint(-12, 12, (P, 1), generator=g).float())   # ranks of different magnitude
    x = torch.randn(P, n, generator=g) * scale
    return [x[r].to(torch.bfloat16) if in_bf16 else x[r].clone() for r in range(P)]


def oracle_in(ts):
    return [bits(t) if t.dtype == torch.bfloat16 else t.numpy() for t in ts]


@pytest.mark.parametrize("P", [1, 2, 5, 8, 64, 127, 128])
@pytest.mark.parametrize("n", [1, 7, 8, 1000, (1 << 20) + 3])
@pytest.mark.parametrize("in_bf16,out_bf16", [(True, True), (True, False), (False, False), (False, True)])
def test_matches_oracle_bit_for_bit(P, n, in_bf16, out_bf16):
    ts = slices_of(P, n, in_bf16, P * 131 + n)
    out = torch.full((n,), float("nan"), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=DEV)
    gtp.gtp_rs_local_sum([t.to(DEV) for t in ts], out)
    torch.cuda.synchronize()
    ref = R.local_sum(oracle_in(ts), out_bf16)
    got = bits(out) if out_bf16 else out.cpu().numpy()
    assert np.array_equal(got.view(np.uint16 if out_bf16 else np.uint32), ref.view(np.uint16 if out_bf16 else np.uint32))


def test_specials_and_in_place():
    """NaN and Inf propagate, fp32 overflow goes to Inf before the cast, and the output may
    be slice 0 itself."""
    vals = np.array([np.nan, np.inf, -np.inf, 3.0e38, 1.0, -0.0, 1e-40, 2.0 ** -130], np.float32)
    a = torch.from_numpy(np.tile(vals, 4))
    b = torch.from_numpy(np.tile(np.array([1.0, -np.inf, 1.0, 3.0e38, -1.0, -0.0, 1e-40, 0.0], np.float32), 4))
    for dt in (torch.float32, torch.bfloat16):
        ts = [a.to(dt), b.to(dt), a.to(dt)]
        dev = [t.to(DEV) for t in ts]
        gtp.gtp_rs_local_sum(dev, dev[0])                     # in place into slice 0
        torch.cuda.synchronize()
        ref = R.local_sum(oracle_in(ts), dt == torch.bfloat16)
        if dt == torch.bfloat16:
            got_v, ref_v = F.bf16_bits_to_f64(bits(dev[0])), F.bf16_bits_to_f64(ref)
            got_b, ref_b = bits(dev[0]), ref
        else:
            got_v, ref_v = dev[0].cpu().numpy(), ref
            got_b, ref_b = got_v.view(np.uint32), ref.view(np.uint32)
        nan = np.isnan(ref_v)
        assert np.array_equal(np.isnan(got_v), nan)          # a NaN is a NaN, whatever its payload
        assert np.array_equal(got_b[~nan], ref_b[~nan])       # everything else bit for bit


def test_7b_bucket_shard_full_size():
    """The 7B buffer's reduce-scatter at full size ([BUF] §8 ledger: 64M-element buckets,
    dp 64, a 1M-element shard a rank): 64 received bf16 slices of 1,000,000 elements summed
    to a bf16 shard, bit for bit."""
    P, n = 64, 1_000_000
    g = W.generator(77, DEV)
    dev = [W.randn_bf16((n,), 1e-3, g, DEV) for _ in range(P)]
    out = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    gtp.gtp_rs_local_sum(dev, out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), R.local_sum([bits(t) for t in dev], True))


def test_receive_buffer_as_one_tensor():
    """The all-to-all's receive buffer passed whole ([P, n], row r from rank r): the same
    shard as the list of its rows, 16-byte-aligned rows (n a multiple of 8 for bf16)."""
    P, n = 16, 4096 + 8
    g = W.generator(91, DEV)
    buf = W.randn_bf16((P, n), 1.0, g, DEV)
    a = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    b = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    gtp.gtp_rs_local_sum(buf, a)
    gtp.gtp_rs_local_sum([buf[r] for r in range(P)], b)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert np.array_equal(bits(a), R.local_sum([bits(buf[r]) for r in range(P)], True))
