"""The hot path is capturable into a CUDA graph (GPU).

One small training step -- zero_grad, two microbatches of fprop / dgrad on the compute
stream and wgrad-accumulate into the flat buffer on a side stream, the gradient norm and
clip coefficient, the fused AdamW sweep, an MXFP8 quantize and MXFP8 forward -- is run
eagerly, then captured into a graph and replayed from the same starting state.  Every
output must match bit for bit: the launches carry their arguments by value and none of
them allocates, synchronises or reads host memory after enqueue.  (The shapes keep every
wgrad contraction unsplit, so no result depends on the order of reduce-adds.)
"""
import pytest
import torch

import param_buffers_gb300 as gtp
from param_buffers_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
M = 128                      # tokens per microbatch: 2 k-blocks, an unsplit wgrad
SHAPES = ((512, 256), (256, 512))


def make_state():
    g = W.generator(11)
    numel = sum(n * k for n, k in SHAPES)
    s = {
        "master": (torch.randn(numel, generator=g) * 0.02).to(DEV),
        "m": torch.zeros(numel, device=DEV),
        "v": torch.zeros(numel, device=DEV),
        "grad": torch.full((numel,), float("nan"), device=DEV),
        "param": torch.empty(numel, dtype=torch.bfloat16, device=DEV),
        "X": [[W.randn_bf16((M, k), 1.0, g).to(DEV) for _, k in SHAPES] for _ in range(2)],
        "dY": [[W.randn_bf16((M, n), 1.0, g).to(DEV) for n, _ in SHAPES] for _ in range(2)],
        "Y": [torch.empty(M, n, dtype=torch.bfloat16, device=DEV) for n, _ in SHAPES],
        "dX": [torch.empty(M, k, dtype=torch.bfloat16, device=DEV) for _, k in SHAPES],
        "ws": torch.empty(1 << 16, dtype=torch.uint8, device=DEV),
        "sumsq": torch.empty(2, dtype=torch.float64, device=DEV),
        "nonfinite": torch.empty(2, dtype=torch.int32, device=DEV),
        "norm": torch.empty(1, device=DEV),
        "clip": torch.empty(1, device=DEV),
        "wq": torch.empty(SHAPES[0], dtype=torch.uint8, device=DEV),
        "ws8": torch.empty(SHAPES[0][0], SHAPES[0][1] // 32, dtype=torch.uint8, device=DEV),
        "xq": torch.empty(M, SHAPES[0][1], dtype=torch.uint8, device=DEV),
        "xs8": torch.empty(M, SHAPES[0][1] // 32, dtype=torch.uint8, device=DEV),
        "y8": torch.empty(M, SHAPES[0][0], dtype=torch.bfloat16, device=DEV),
    }
    s["param"].copy_(s["master"].to(torch.bfloat16))
    return s


def step(s, side):
    offsets = [0, SHAPES[0][0] * SHAPES[0][1]]
    buckets = [{"offset": 0, "numel": offsets[1]}, {"offset": offsets[1], "numel": s["grad"].numel() - offsets[1]}]
    factors = [0.5, 0.5]
    gtp.gtp_buffer_zero(s["grad"])
    for mb in range(2):
        start = torch.cuda.Event()
        start.record()
        side.wait_event(start)
        for i, (n, k) in enumerate(SHAPES):
            Wv = s["param"][offsets[i]:offsets[i] + n * k].view(n, k)
            gtp.gtp_linear_fprop(s["X"][mb][i], Wv, s["Y"][i])
            gtp.gtp_linear_dgrad(s["dY"][mb][i], Wv, s["dX"][i])
            with torch.cuda.stream(side):
                gtp.gtp_linear_wgrad_accum(s["dY"][mb][i], s["X"][mb][i], s["grad"], offsets[i])
        done = torch.cuda.Event()
        done.record(side)
        torch.cuda.current_stream().wait_event(done)
    gtp.gtp_grad_norm(s["grad"], buckets, factors, 1.0, s["ws"], s["sumsq"], s["nonfinite"], s["norm"], s["clip"])
    gtp.gtp_adam_step_flat(s["grad"], s["master"], s["m"], s["v"], s["param"], buckets, factors,
                           gtp.AdamHparams(), step=1, grad_scale=s["clip"])
    gtp.gtp_mxfp8_quantize_rowwise(s["master"][:offsets[1]].view(SHAPES[0]), s["wq"], s["ws8"])
    gtp.gtp_mxfp8_quantize_rowwise(s["X"][0][0], s["xq"], s["xs8"])
    gtp.gtp_linear_fprop_mxfp8(s["xq"], s["xs8"], s["wq"], s["ws8"], s["y8"])


def snapshot(s):
    out = {}
    for k, v in s.items():
        if isinstance(v, torch.Tensor):
            out[k] = v.detach().clone()
        elif k in ("Y", "dX"):
            out[k] = [t.detach().clone() for t in v]
    return out


def restore(s, snap):
    for k, v in snap.items():
        if isinstance(v, list):
            for t, u in zip(s[k], v):
                t.copy_(u)
        else:
            s[k].copy_(v)


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_layer_step_replays_bit_exact_from_a_cuda_graph():
    s = make_state()
    side = torch.cuda.Stream()
    step(s, side)                       # warm-up: one-time kernel configuration happens here
    torch.cuda.synchronize()
    s0 = make_state()
    for k, v in s0.items():             # same starting point for both runs
        if isinstance(v, torch.Tensor):
            s[k].copy_(v)
    init = snapshot(s)
    step(s, side)
    torch.cuda.synchronize()
    eager = snapshot(s)

    restore(s, init)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=cap):
        step(s, side)
    torch.cuda.synchronize()
    restore(s, init)                    # capture launches nothing, but start clean regardless
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    replay = snapshot(s)

    for k in ("master", "m", "v", "param", "grad", "sumsq", "nonfinite", "norm", "clip", "wq", "ws8", "y8"):
        assert bits_equal(eager[k], replay[k]), k
    for k in ("Y", "dX"):
        for a, b in zip(eager[k], replay[k]):
            assert bits_equal(a, b), k
    assert torch.isfinite(replay["norm"]).all() and replay["norm"].item() > 0
