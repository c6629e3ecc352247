"""Failure detection of the tensor-core kernels' waits, exercised without a fault (GPU).

Every mbarrier wait in the library's kernels gives up after a time limit, raises a bit in
a per-device word and lets the kernel return.  gtp_selftest_wait_timeout runs that same
bounded wait, with a 1 ms limit, on an mbarrier that nothing arrives on: the wait must
run out (the kernel lasts at least the limit and far less than a second), the bit must
be reported by gtp_wait_timeouts, and the context must keep working - a GEMM launched
afterwards still matches the oracle and reports no expired wait of its own.
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
SELFTEST_BIT = 0x100


def bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def test_expired_wait_is_reported_and_the_context_survives():
    gtp.gtp_wait_timeouts(reset=True)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    gtp.gtp_selftest_wait_timeout(1_000_000)          # 1 ms
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e)
    assert 1.0 <= ms < 1000.0, ms                     # the wait lasted its limit, then returned
    flags = gtp.gtp_wait_timeouts(reset=True)
    assert flags & SELFTEST_BIT, hex(flags)
    assert gtp.gtp_wait_timeouts() == 0               # reset took effect

    # the context keeps working: a GEMM after the expired wait is correct and clean
    M, N, K = 300, 520, 200
    X, Wt, dY = W.linear_inputs(M, N, K, W.generator(77))
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    gtp.gtp_linear_fprop(X.to(DEV), Wt.to(DEV), Y)
    torch.cuda.synchronize()
    ref = G.fprop(bits(X), bits(Wt))
    got = F.bf16_bits_to_f64(bits(Y))
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 2e-3
    assert gtp.gtp_wait_timeouts() == 0


def test_selftest_twice_in_a_row():
    """Two expired waits back to back: each returns, the bit is set once more after a reset."""
    for _ in range(2):
        gtp.gtp_wait_timeouts(reset=True)
        gtp.gtp_selftest_wait_timeout(100_000)        # 100 us
        torch.cuda.synchronize()
        assert gtp.gtp_wait_timeouts(reset=True) & SELFTEST_BIT
