#!/usr/bin/env python3
"""Benchmark of the hot path on one GB300 (or N independent replicas under torchrun).

One step = one pass of the whole path over one batch of synthetic input, for one
Llama-3.2-1B layer at TP=2 (h 2048, f 8192, 32/8 heads, d_h 64), seq 8192 x micro-batch 1:
  zero_grad_buffer (grad_data = 0)
  8 microbatches x {QKV [1536,2048], O [2048,1024], fc1 [8192,2048], fc2 [2048,4096]}:
      fprop Y = X W^T, dgrad dX = dY W, wgrad main_grad += dY^T X into the flat fp32 buffer
  grad norm + clip coefficient (max_norm 1.0)
  the fused sweep over the flat buffer: bucket scale -> clip -> AdamW -> bf16 cast -> zero
  the MXFP8 write of the fc1/fc2 masters and one MXFP8 fc1 forward
The weights are views of the bf16 param_data buffer and main_grad views of grad_data, at
the offsets the layout engine assigns (30,412,800 elements, one 40M bucket, dp = 2).
The GEMMs keep the layer's dependencies (forward chain, then the dgrad chain in reverse);
by default (--schedule overlap) each launch groups one linear's backward of microbatch i
(dgrad + wgrad accumulate) with one linear's forward of microbatch i+1, so that the two
chains advance together; the other schedules launch every GEMM alone or each backward as
one launch (LayerStep).

value = bf16 GEMM TFLOP/s of the whole step (11.96 TFLOP per step / step time).  Also
reported: the fused AdamW sweep (bf16 and native-MXFP8 variants) alone on the 7B-style
flat buffer (1.875e9 elements) in GB/s, the block-scaled GEMMs alone on the fc1 shape,
and the end-to-end step with host inputs (e2e).  --impl reference times the CPU oracle
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "wgrad-accum GEMM TFLOP/s (% bf16 peak); flat-buffer AdamW GB/s (% HBM peak)"
SCHEDULES = ("separate", "one-stream", "grouped", "overlap")
SWEEP_BYTES_PER_ELEM = 34   # read g, p, m, v (16) + write p, m, v (12), bf16 param (2), zero g (4)
SWEEP_MX_BYTES_PER_ELEM = 33.03125   # the same with E4M3 (1) + E8M0 (1/32) written instead of bf16
SWEEP_BF16_GRAD_BYTES_PER_ELEM = 30  # a bf16 grad buffer: read g (2), zero g (2) instead of 4 + 4
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gtp", "reference"], default="gtp")
    ap.add_argument("--e2e-steps", type=int, default=5, help="steps in each of the e2e loop's repetitions")
    ap.add_argument("--e2e-reps", type=int, default=15, help="timed repetitions of the e2e loop")
    ap.add_argument("--copy-streams", type=int, default=2, help="host-to-device copy streams of the e2e run")
    ap.add_argument("--schedule", choices=SCHEDULES, default="overlap",
                    help="how the step launches its GEMMs (see LayerStep)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["fprop", "dgrad", "wgrad", "wgrad_det", "backward", "overlap", "adam", "adam_mx", "gradnorm", "mxfp8_fprop", "mxfp8_dgrad", "mxfp8_wgrad",
                                       "nvfp4_fprop", "mxfp8_fprop_tiled", "nvfp4_fprop_tiled", "mxfp8_dgrad_tiled",
                                       "mxfp8_wgrad_tiled", "quantize_mxfp8_rowwise",
                                       "quantize_mxfp8_columnwise", "quantize_mxfp8_columnwise_group",
                                       "quantize_mxfp8_rowwise_group", "rs_local_sum",
                                       "quantize_nvfp4_rowwise"], default=None,
                    help="profiling mode: launch one kernel of the step, warmup + steps times")
    ap.add_argument("--linear", default="fc1", help="the layer linear used by --only (overlap: BWD+FWD, e.g. fc1+proj)")
    ap.add_argument("--sweep-numel", type=int, default=30_412_800,
                    help="buffer elements of --only adam / adam_mx / gradnorm (default: the layer buffer)")
    ap.add_argument("--summarize-launches", metavar="CSV", default=None,
                    help="print per-kernel launches / time / share from an ncu --csv launch list and exit")
    ap.add_argument("--source-hash", action="store_true", help="print the GEMM source hash used by profiles/traffic.txt")
    return ap.parse_args()


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms; only samples inside [t0, t1] are kept."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.lines: list[tuple[float, str]] = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        sm, mx, reasons, n = [], 0.0, set(), 0
        for ts, line in self.lines:
            if not (t0 - 0.25 <= ts <= t1 + 0.25):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            n += 1
            try:
                sm.append(float(f[2]))
                mx = max(mx, float(f[3]))
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), f[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx or None, "reasons": sorted(reasons),
                "samples": n}


class NvmlClockSampler:
    """SM clock, power and clock-event reasons read through NVML (read-only queries) every
    `period_s` seconds, so that a timed region of a fraction of a second still holds tens of
    samples; same summary as ClockSampler.  Raises OSError when NVML cannot be loaded."""
    # public NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.01):
        import ctypes as C
        nvml = None
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                nvml = C.CDLL(name)
                break
            except OSError:
                continue
        if nvml is None or nvml.nvmlInit_v2() != 0:
            raise OSError("NVML unavailable")
        self.C, self.nvml = C, nvml
        self.handle = self._handle(device_index)
        self.samples: list[tuple[float, float, float, float, int]] = []
        mx = C.c_uint(0)
        self.max_mhz = float(mx.value) if nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, C.byref(mx)) == 0 else None
        try:
            self.reasons_fn = nvml.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self.reasons_fn = nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        self.period = period_s
        self.running = True
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _handle(self, device_index: int):
        """The NVML handle of the CUDA device (by UUID, which CUDA_VISIBLE_DEVICES does not renumber)."""
        C, nvml = self.C, self.nvml
        h = C.c_void_p()
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            for key in (f"GPU-{uuid}", uuid):
                if nvml.nvmlDeviceGetHandleByUUID(key.encode(), C.byref(h)) == 0:
                    return h
        except Exception:
            pass
        if nvml.nvmlDeviceGetHandleByIndex_v2(device_index, C.byref(h)) != 0:
            raise OSError("NVML device handle")
        return h

    def _run(self):
        C, nvml, h = self.C, self.nvml, self.handle
        clk, pw, rs = C.c_uint(0), C.c_uint(0), C.c_ulonglong(0)
        while self.running:
            ok = nvml.nvmlDeviceGetClockInfo(h, 1, C.byref(clk)) == 0       # NVML_CLOCK_SM
            nvml.nvmlDeviceGetPowerUsage(h, C.byref(pw))
            self.reasons_fn(h, C.byref(rs))
            if ok:
                self.samples.append((time.time(), float(clk.value), pw.value / 1000.0, 0.0, int(rs.value)))
            time.sleep(self.period)

    def stop(self):
        self.running = False
        self.thread.join(timeout=1.0)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        sm = sorted(x[1] for x in inside)
        reasons = sorted({name for x in inside for bit, name in self.REASONS.items() if x[4] & bit})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(inside), "sm_mhz_min": sm[0] if sm else None,
                "power_w_max": max((x[2] for x in inside), default=None),
                "source": f"nvml, {self.period * 1e3:g} ms"}


def clock_sampler(device_index: int, period_s: float = 0.01):
    try:
        return NvmlClockSampler(device_index, period_s)
    except (OSError, AttributeError):
        return ClockSampler(device_index)


# ----------------------------------------------------------------------------- workload

class LayerStep:
    """Device-resident state of the layer workload and the step that runs through the C ABI."""

    def __init__(self, device, seed_offset: int = 0, schedule: str = "overlap"):
        import torch
        import param_buffers_gb300 as gtp
        from param_buffers_gb300 import workloads as W
        self.torch, self.gtp, self.W = torch, gtp, W
        self.dev = device
        # How the GEMMs of a microbatch are launched; every schedule keeps the layer's own
        # dependencies (the forward chain qkv -> proj -> fc1 -> fc2, the backward chain of
        # dgrads in reverse) and does the same products:
        #   separate    each GEMM its own launch; a microbatch's wgrads on a side stream,
        #               overlapping the dgrads (a wgrad needs X and dY, a dgrad dY and W)
        #   one-stream  each GEMM its own launch, all on one stream
        #   grouped     each linear's backward (dgrad + wgrad accumulate) as one launch
        #   overlap     microbatch i's backward of one linear grouped, in one launch, with
        #               microbatch i+1's forward of another: the two chains advance together
        #               (they share only the weights, which do not change while gradients
        #               accumulate)
        self.schedule = schedule
        self.side = torch.cuda.Stream(device) if schedule == "separate" else None
        self.side_done = [torch.cuda.Event() for _ in range(W.LAYER_MICROBATCHES)]
        bw = W.layer_buffer()
        self.bw = bw
        self.lay = gtp.gtp_buffer_layout([gtp.ParamDesc(p.numel, p.dtype) for p in bw.params],
                                         gtp.LayoutConfig(bw.bucket_size, bw.dp_size, True))
        self.numel = self.lay.buffers[0]["numel"]
        assert self.numel == LAYER_BUFFER_NUMEL, self.numel
        self.factors = [bw.gradient_scaling_factor] * len(self.lay.buckets)
        self.hp = gtp.AdamHparams(**bw.hparams)
        g = W.generator(W.seed_of("layer") + seed_offset, device)
        self.grad, self.master, self.m, self.v, self.param = W.buffer_state(self.numel, g, device)
        names = [p.name for p in bw.params]
        self.offsets = {lin.name: self.lay.index[names.index(lin.name)]["start"] for lin in W.LAYER_LINEARS}
        self.M = W.LAYER_M
        self.lins = W.LAYER_LINEARS
        self.X, self.dY = [], []
        for _ in range(W.LAYER_MICROBATCHES):
            self.X.append({l.name: W.randn_bf16((self.M, l.K), 1.0, g, device) for l in self.lins})
            self.dY.append({l.name: W.randn_bf16((self.M, l.N), 1.0, g, device) for l in self.lins})
        self.Y = {l.name: torch.empty(self.M, l.N, dtype=torch.bfloat16, device=device) for l in self.lins}
        self.dX = {l.name: torch.empty(self.M, l.K, dtype=torch.bfloat16, device=device) for l in self.lins}
        # Low-precision weight path: the updated fp32 masters of the FFN weights are written
        # as MXFP8 once per step, and fc1's forward runs on the block-scaled tensor cores
        # (microbatch 0's activations, quantized rowwise along K).
        self.mx_lins = [l for l in self.lins if l.name in ("fc1", "fc2")]
        self.mx_q = {l.name: torch.empty(l.N, l.K, dtype=torch.uint8, device=device) for l in self.mx_lins}
        # scales in the tiled layout (the tensor core's read order; the tiled forward fetches a
        # stage's scales as three contiguous copies)
        self.mx_s = {l.name: torch.empty(gtp.gtp_sf_tiled_bytes(l.N, l.K // 32), dtype=torch.uint8, device=device)
                     for l in self.mx_lins}
        fc1 = next(l for l in self.lins if l.name == "fc1")
        self.fc1 = fc1
        self.xq = torch.empty(self.M, fc1.K, dtype=torch.uint8, device=device)
        self.xs = torch.empty(gtp.gtp_sf_tiled_bytes(self.M, fc1.K // 32), dtype=torch.uint8, device=device)
        self.y_mx = torch.empty(self.M, fc1.N, dtype=torch.bfloat16, device=device)
        # Gradient norm, non-finite check and the --clip-grad 1.0 coefficient, which the
        # sweep applies from the device.
        nb = len(self.lay.buckets)
        self.norm_ws = torch.empty(max(16, gtp.gtp_grad_norm_workspace_bytes(self.lay.c_buckets)), dtype=torch.uint8,
                                   device=device)
        self.sumsq = torch.empty(nb, dtype=torch.float64, device=device)
        self.nonfinite = torch.empty(nb, dtype=torch.int32, device=device)
        self.total_norm = torch.empty(1, dtype=torch.float32, device=device)
        self.clip_coef = torch.empty(1, dtype=torch.float32, device=device)
        self.t = 0
        self.grad_zeroed = False  # buffer_state's grad is not zero
        self.flops = 3 * W.LAYER_MICROBATCHES * sum(W.linear_flops(self.M, l.N, l.K) for l in self.lins)
        self.mx_flops = W.linear_flops(self.M, fc1.N, fc1.K)
        nmb, nl = W.LAYER_MICROBATCHES, len(self.lins)
        gemm_launches = {"separate": 3 * nmb * nl, "one-stream": 3 * nmb * nl, "grouped": 2 * nmb * nl,
                         "overlap": nl + nmb * nl}[schedule]
        # a step after a sweep: GEMMs, grad norm (2), sweep, the grouped MXFP8 quantize, MXFP8 forward
        self.launches_per_step = gemm_launches + 2 + 1 + 1 + 1
        # FLOPs of one launch of each timed kind (the per-kernel table and the roofline)
        lf = {l.name: W.linear_flops(self.M, l.N, l.K) for l in self.lins}
        self.kind_flops = {}
        for l in self.lins:
            for k in ("fprop", "dgrad", "wgrad"):
                self.kind_flops[(k, l.name)] = lf[l.name]
            self.kind_flops[("backward", l.name)] = 2 * lf[l.name]
        for lb, lfw in zip(reversed(self.lins), self.lins):
            self.kind_flops[("overlap", f"{lb.name}+{lfw.name}")] = 2 * lf[lb.name] + lf[lfw.name]

    def weight(self, lin):
        o = self.offsets[lin.name]
        return self.param[o:o + lin.N * lin.K].view(lin.N, lin.K)

    def input_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for d in (*self.X, *self.dY) for t in d.values())

    def run(self, timer=None):
        for _, op in self.plan():
            op(timer)

    def plan(self):
        """The step as a list of (microbatch whose inputs the launches need, or None;
        op(timer) that enqueues them)."""
        nmb = len(self.X)
        ops = [(None, self.begin)]
        if self.schedule == "overlap":
            ops.append((0, lambda timer: self.forward(0, timer)))
            for mb in range(nmb):
                nxt = mb + 1 if mb + 1 < nmb else None
                ops.append((mb if nxt is None else nxt, lambda timer, mb=mb, nxt=nxt: self.overlapped(mb, nxt, timer)))
        else:
            for mb in range(nmb):
                ops.append((mb, lambda timer, mb=mb: self.microbatch(mb, timer)))
        ops.append((None, self.finish))
        return ops

    def forward(self, mb: int, timer=None):
        for lin in self.lins:
            self._call(timer, ("fprop", lin.name), self.gtp.gtp_linear_fprop, self.X[mb][lin.name], self.weight(lin),
                       self.Y[lin.name])

    def overlapped(self, mb: int, nxt, timer=None):
        """Microbatch mb's backward, linear by linear in reverse, each grouped in one launch
        with microbatch nxt's forward of the linear at the same position of the forward
        chain (nxt None: the backward alone)."""
        gtp = self.gtp
        for lb, lfw in zip(reversed(self.lins), self.lins):
            X, dY, Wb = self.X[mb][lb.name], self.dY[mb][lb.name], self.weight(lb)
            descs = [gtp.gemm_desc("dgrad", dY, Wb, self.dX[lb.name]),
                     gtp.gemm_desc("wgrad", dY, X, self.grad, self.offsets[lb.name])]
            if nxt is None:
                self._call(timer, ("backward", lb.name), gtp.gtp_linear_grouped, descs)
            else:
                descs.append(gtp.gemm_desc("fprop", self.X[nxt][lfw.name], self.weight(lfw), self.Y[lfw.name]))
                self._call(timer, ("overlap", f"{lb.name}+{lfw.name}"), gtp.gtp_linear_grouped, descs)

    @staticmethod
    def _call(timer, kind, fn, *a, **k):
        if timer is None:
            fn(*a, **k)
        else:
            timer.around(kind, lambda: fn(*a, **k))

    def begin(self, timer=None):
        """The head of a step.  grad_data must be zero before the first accumulate: the
        fused sweep zeroes it at the end of every step (the pages' iteration-start
        zero_grad_buffer, fused into the sweep as A5), so only a step that follows no sweep
        -- the first -- launches the standalone zero."""
        self.t += 1
        if not self.grad_zeroed:
            self._call(timer, "zero", self.gtp.gtp_buffer_zero, self.grad)
        self.grad_zeroed = False  # the accumulates fill it

    def microbatch(self, mb: int, timer=None):
        """fprop, dgrad and wgrad-accumulate of the four linears on microbatch mb."""
        gtp, torch = self.gtp, self.torch
        if self.schedule == "grouped":
            # forward of the four linears, then each linear's backward as one launch, in reverse
            for lin in self.lins:
                self._call(timer, ("fprop", lin.name), gtp.gtp_linear_fprop, self.X[mb][lin.name], self.weight(lin),
                           self.Y[lin.name])
            for lin in reversed(self.lins):
                self._call(timer, ("backward", lin.name), gtp.gtp_linear_backward, self.dY[mb][lin.name],
                           self.X[mb][lin.name], self.weight(lin), self.dX[lin.name], self.grad,
                           self.offsets[lin.name])
            return
        if self.side is None:
            for lin in self.lins:
                Wv = self.weight(lin)
                X, dY = self.X[mb][lin.name], self.dY[mb][lin.name]
                self._call(timer, ("fprop", lin.name), gtp.gtp_linear_fprop, X, Wv, self.Y[lin.name])
                self._call(timer, ("dgrad", lin.name), gtp.gtp_linear_dgrad, dY, Wv, self.dX[lin.name])
                self._call(timer, ("wgrad", lin.name), gtp.gtp_linear_wgrad_accum, dY, X, self.grad,
                           self.offsets[lin.name])
            return
        # forward of the four linears, then the backward in reverse order: dgrads on the
        # compute stream, wgrads on the side stream once the microbatch's inputs are there
        start = torch.cuda.Event()
        start.record()
        self.side.wait_event(start)
        for lin in self.lins:
            self._call(timer, ("fprop", lin.name), gtp.gtp_linear_fprop, self.X[mb][lin.name], self.weight(lin),
                       self.Y[lin.name])
        for lin in reversed(self.lins):
            X, dY = self.X[mb][lin.name], self.dY[mb][lin.name]
            self._call(timer, ("dgrad", lin.name), gtp.gtp_linear_dgrad, dY, self.weight(lin), self.dX[lin.name])
            with torch.cuda.stream(self.side):
                self._call(timer, ("wgrad", lin.name), gtp.gtp_linear_wgrad_accum, dY, X, self.grad,
                           self.offsets[lin.name])
        self.side_done[mb].record(self.side)
        torch.cuda.current_stream().wait_event(self.side_done[mb])  # the microbatch ends when its wgrads do

    def finish(self, timer=None):
        """The optimizer step: grad norm and clip coefficient, the fused AdamW sweep, the
        MXFP8 write of the FFN masters, and one MXFP8 forward (microbatch 0's fc1 input)."""
        gtp, call = self.gtp, self._call
        if self.side is not None:  # every wgrad has landed in grad_data
            self.torch.cuda.current_stream().wait_stream(self.side)
        call(timer, "gradnorm", gtp.gtp_grad_norm, self.grad, self.lay.c_buckets, self.factors, 1.0, self.norm_ws,
             self.sumsq, self.nonfinite, self.total_norm, self.clip_coef)
        call(timer, "adam", gtp.gtp_adam_step_flat, self.grad, self.master, self.m, self.v, self.param,
             self.lay.c_buckets, self.factors, self.hp, step=self.t, grad_scale=self.clip_coef)
        self.grad_zeroed = bool(self.hp.zero_grad_after)
        views = [(self.master[self.offsets[l.name]:self.offsets[l.name] + l.N * l.K].view(l.N, l.K),
                  self.mx_q[l.name], self.mx_s[l.name]) for l in self.mx_lins]
        views.append((self.X[0]["fc1"], self.xq, self.xs))
        call(timer, "quant", gtp.gtp_mxfp8_quantize_rowwise_group, views)   # one launch for the three
        call(timer, "mxfp8", gtp.gtp_linear_fprop_mxfp8_tiled, self.xq, self.xs, self.mx_q["fc1"], self.mx_s["fc1"],
             self.y_mx)


class KernelTimer:
    """CUDA events around every launch on the launching stream; totals per kernel kind."""

    def __init__(self, torch):
        self.torch = torch
        self.events: list[tuple[object, object, object]] = []

    def around(self, kind, fn):
        s = self.torch.cuda.Event(enable_timing=True)
        e = self.torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        self.events.append((kind, s, e))

    def totals(self) -> dict:
        out: dict = {}
        for kind, s, e in self.events:
            out.setdefault(kind, [0.0, 0])
            out[kind][0] += s.elapsed_time(e)
            out[kind][1] += 1
        return out


def time_sweep_7b(torch, gtp, W, device, reps: int = 10) -> dict:
    """The fused AdamW sweep alone on the 1.875e9-element buffer (L2 is 129 MB: every
    launch streams 63.75 GB from HBM)."""
    bw = W.seven_b_buffer()
    lay = gtp.gtp_buffer_layout([gtp.ParamDesc(p.numel, p.dtype, is_shared_embedding=p.is_shared_embedding)
                                 for p in bw.params], gtp.LayoutConfig(bw.bucket_size, bw.dp_size, True))
    n = lay.buffers[0]["numel"]
    g = W.generator(W.seed_of("7b"), device)
    grad, master, m, v, param = W.buffer_state(n, g, device)
    fac = [bw.gradient_scaling_factor] * len(lay.buckets)
    hp = gtp.AdamHparams(**bw.hparams)          # the full sweep, zeroing included (34 B/element)
    for t in range(3):
        gtp.gtp_adam_step_flat(grad, master, m, v, param, lay.c_buckets, fac, hp, step=t + 1)
    torch.cuda.synchronize()

    def timed(call, first_step):
        ts = []
        for t in range(reps):
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record()
            call(first_step + t)
            e.record()
            e.synchronize()
            ts.append(s.elapsed_time(e))
        return sum(ts) / len(ts)

    ms = timed(lambda t: gtp.gtp_adam_step_flat(grad, master, m, v, param, lay.c_buckets, fac, hp, step=t), 4)
    del param
    # the same buffer as native MXFP8 parameters: the sweep writes E4M3 codes + E8M0 scales
    q = torch.empty(n, dtype=torch.uint8, device=device)
    sc = torch.empty(n // 32, dtype=torch.uint8, device=device)
    for t in range(3):
        gtp.gtp_adam_step_flat_mxfp8(grad, master, m, v, q, sc, lay.c_buckets, fac, hp, step=reps + 4 + t)
    torch.cuda.synchronize()
    ms_mx = timed(lambda t: gtp.gtp_adam_step_flat_mxfp8(grad, master, m, v, q, sc, lay.c_buckets, fac, hp, step=t),
                  reps + 7)
    del q, sc
    # the same sweep over a bf16 grad buffer (grad_reduce_in_fp32 off): 30 B/element
    gb = grad.to(torch.bfloat16)
    pb = torch.empty(n, dtype=torch.bfloat16, device=device)
    for t in range(3):
        gtp.gtp_adam_step_flat(gb, master, m, v, pb, lay.c_buckets, fac, hp, step=2 * reps + 7 + t)
    torch.cuda.synchronize()
    ms_bg = timed(lambda t: gtp.gtp_adam_step_flat(gb, master, m, v, pb, lay.c_buckets, fac, hp, step=t),
                  2 * reps + 10)
    del gb, pb
    q = sc = None
    # the gradient-norm pass (one read of grad_data, per-bucket sums of squares) on the same buffer
    nb = len(lay.buckets)
    ws = torch.empty(max(16, gtp.gtp_grad_norm_workspace_bytes(lay.c_buckets)), dtype=torch.uint8, device=device)
    outs = (torch.empty(nb, dtype=torch.float64, device=device), torch.empty(nb, dtype=torch.int32, device=device),
            torch.empty(1, device=device), torch.empty(1, device=device))
    norm = lambda t: gtp.gtp_grad_norm(grad, lay.c_buckets, fac, 1.0, ws, *outs)
    for _ in range(3):
        norm(0)
    torch.cuda.synchronize()
    ms_norm = batch_ms(torch, norm, reps, per_batch=5)
    del grad, master, m, v, q, sc, ws, outs
    torch.cuda.empty_cache()
    rs = time_rs_local_sum(torch, gtp, W, device)
    return {"numel": n, "ms": ms, "gbs": SWEEP_BYTES_PER_ELEM * n / ms / 1e6, "launches": reps,
            "mxfp8": {"ms": ms_mx, "bytes_per_elem": SWEEP_MX_BYTES_PER_ELEM,
                      "gbs": SWEEP_MX_BYTES_PER_ELEM * n / ms_mx / 1e6, "launches": reps},
            "grad_norm": {"ms": ms_norm, "bytes_per_elem": 4, "gbs": 4 * n / ms_norm / 1e6, "launches": reps},
            "bf16_grad": {"ms": ms_bg, "bytes_per_elem": SWEEP_BF16_GRAD_BYTES_PER_ELEM,
                          "gbs": SWEEP_BF16_GRAD_BYTES_PER_ELEM * n / ms_bg / 1e6, "launches": reps},
            "rs_local_sum": rs}


def time_rs_local_sum(torch, gtp, W, device, P: int = 64, n: int = 1_000_000, reps: int = 30) -> dict:
    """The local fp32 sum of the all-to-all reduce-scatter for one bucket of the 7B buffer
    (64M-element buckets at dp 64: 64 received bf16 slices of a 1M-element shard, summed
    into a bf16 shard), rotating over three sets of slices (384 MB, more than L2).  Bytes
    are algorithmic: P slices read once, the shard written."""
    g = W.generator(W.seed_of("7b") + 3, device)
    # each set is one all-to-all receive buffer, [P, n]: row r came from rank r
    sets = [W.randn_bf16((P, n), 1e-3, g, device) for _ in range(3)]
    outs = [torch.empty(n, dtype=torch.bfloat16, device=device) for _ in range(3)]
    fn = lambda t: gtp.gtp_rs_local_sum(sets[t % 3], outs[t % 3])
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    ms = batch_ms(torch, fn, reps, per_batch=6)
    nbytes = (P + 1) * 2 * n
    del sets, outs
    torch.cuda.empty_cache()
    return {"slices": P, "shard_elems": n, "ms": ms, "bytes": nbytes, "gbs": nbytes / ms / 1e6, "launches": reps}


# ----------------------------------------------------------------------------- oracle timing

# elements of the layer's flat param/grad buffer (the dist-opt layout of its six
# parameters, one bucket); the timed step checks it against the library's layout
LAYER_BUFFER_NUMEL = 30_412_800


def oracle_sample(seconds: float = 10.0, seed: int = 0) -> dict:
    """The CPU oracle as it stands on a bounded sample of the layer workload: the three
    GEMMs of all four linears on a slice of tokens of one microbatch, plus the AdamW
    sweep on a slice of the flat buffer.  Repeats until `seconds` have passed."""
    import numpy as np
    import torch
    from oracle import adamw as A
    from oracle import gemm as G
    from param_buffers_gb300 import workloads as W

    Ms = 1024
    g = W.generator(W.seed_of("layer") + 17 + seed)
    data = []
    for lin in W.LAYER_LINEARS:
        X, Wt, dY = W.linear_inputs(Ms, lin.N, lin.K, g)
        data.append(tuple(t.view(torch.int16).numpy().view(np.uint16) for t in (X, Wt, dY)))
    n_sweep = 4_000_000
    grad, master, m, v = (t.numpy() for t in W.buffer_state(n_sweep, g)[:4])
    fac = np.full(n_sweep, 0.5)
    h = A.AdamWHparams()
    flops = sum(3 * 2 * Ms * lin.N * lin.K for lin in W.LAYER_LINEARS)
    t_gemm = t_sweep = 0.0
    reps = 0
    t_start = time.perf_counter()
    while reps == 0 or time.perf_counter() - t_start < seconds:
        t0 = time.perf_counter()
        for (X, Wt, dY) in data:
            G.to_bf16(G.fprop(X, Wt))
            G.to_bf16(G.dgrad(dY, Wt))
            G.wgrad_accum(np.zeros((Wt.shape[0], Wt.shape[1]), np.float32), dY, X)
        t1 = time.perf_counter()
        A.fused_sweep(grad, master, m, v, fac, 1, h)
        t2 = time.perf_counter()
        t_gemm += t1 - t0
        t_sweep += t2 - t1
        reps += 1
    threads = os.cpu_count()
    try:
        from threadpoolctl import threadpool_info
        blas = [i for i in threadpool_info() if i.get("user_api") == "blas"]
        if blas:
            threads = blas[0]["num_threads"]
    except Exception:
        pass
    return {"tflops": flops * reps / t_gemm / 1e12, "sweep_gbs": SWEEP_BYTES_PER_ELEM * n_sweep * reps / t_sweep / 1e9,
            "cores": threads, "reps": reps, "seconds": t_gemm + t_sweep,
            "sample": f"oracle fp64 fprop+dgrad+wgrad of the 4 layer linears on {Ms} of 8192 tokens, "
                      f"and the AdamW sweep on {n_sweep} of {LAYER_BUFFER_NUMEL:,} buffer elements, x{reps}"}


# ----------------------------------------------------------------------------- main

def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if ws > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        pg = dist
    return ws, rank, local, pg


def reduce_max(pg, value: float) -> float:
    """The largest `value` over the ranks (every rank gets it); the launches use NCCL, so
    the tensor lives on the GPU, except over gloo (the CPU tests of this path)."""
    if pg is None:
        return value
    import torch
    dev = "cuda" if pg.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def traffic_from_profiles(kernel: str) -> float | None:
    """dram bytes per launch of `kernel` from the committed ncu summary, if its recorded
    source hash still matches the kernel source."""
    f = ROOT / "profiles" / "traffic.txt"
    if not f.exists():
        return None
    rows = {}
    for line in f.read_text().splitlines():
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#"):
            rows[parts[0]] = (parts[1], parts[2])
    if kernel not in rows:
        return None
    src_hash, traffic = rows[kernel]
    if gemm_source_hash() != src_hash:
        return None
    return float(traffic)


def sweep_traffic_per_elem() -> float | None:
    """DRAM bytes per element of the fused AdamW sweep from the committed ncu summary, if
    its recorded source hash still matches the sweep's sources."""
    f = ROOT / "profiles" / "traffic_sweep.txt"
    if not f.exists():
        return None
    for line in f.read_text().splitlines():
        parts = line.split()
        if len(parts) >= 3 and parts[0] == "adam_flat" and not line.startswith("#"):
            return float(parts[2]) if parts[1] == sweep_source_hash() else None
    return None


def sweep_source_hash() -> str:
    """Hash of the sweep kernel's sources; a traffic figure taken from another version is void."""
    import hashlib
    h = hashlib.sha256()
    for name in ("sweep.cu", "device.h"):
        h.update((ROOT / "param_buffers_gb300" / "csrc" / name).read_bytes())
    return h.hexdigest()[:16]


def gemm_source_hash() -> str:
    """Hash of the bf16 GEMM kernel sources; a traffic figure taken from another version is void."""
    import hashlib
    h = hashlib.sha256()
    for name in ("gemm_bf16.cu", "gemm_common.cuh", "sm100_ptx.cuh", "tensor_map.cu"):
        h.update((ROOT / "param_buffers_gb300" / "csrc" / name).read_bytes())
    return h.hexdigest()[:16]


def layer_config(W, replicas: int, sm_count) -> dict:
    """The layer workload, as both arms name it (`config` of the JSON line)."""
    M, mb = W.LAYER_M, W.LAYER_MICROBATCHES
    flops = 3 * mb * sum(W.linear_flops(M, l.N, l.K) for l in W.LAYER_LINEARS)
    inputs = mb * M * 2 * sum(l.K + l.N for l in W.LAYER_LINEARS)
    return {"workload": "llama3.2-1b layer, TP=2 shard: QKV/O/fc1/fc2 fprop+dgrad+wgrad-accum, "
                        f"{mb} microbatches of seq {M} x mb 1, then the fused AdamW sweep over the "
                        f"{LAYER_BUFFER_NUMEL:,}-element flat buffer, the MXFP8 quantize of the updated fc1/fc2 "
                        "masters and one MXFP8 fc1 forward; value counts the bf16 GEMM FLOPs only",
            "M": M, "microbatches": mb, "gemm_tflop_per_step": flops / 1e12, "flat_buffer_elems": LAYER_BUFFER_NUMEL,
            "l2": f"inputs larger than L2: {inputs / 1e9:.2f} GB of fresh activations per step",
            "replicas": replicas, "sm_count": sm_count}


def run_reference(args, ws, rank):
    if rank != 0:
        return
    import torch
    from param_buffers_gb300 import workloads as W
    # the same config as the timed arm's (the device is only asked for its SM count)
    sm_count = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else None
    results = []
    for _ in range(args.warmup):
        oracle_sample(seconds=0.0)
    for _ in range(args.steps):
        results.append(oracle_sample(seconds=0.0))
    tf = sum(r["tflops"] for r in results) / len(results)
    sample = results[0]["sample"].rsplit(",", 1)[0]
    line = {"impl": "reference", "metric": METRIC, "value": tf, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": layer_config(W, 1, sm_count),
            "cpu_baseline": {"value": tf, "unit": "TFLOP/s", "cores": results[0]["cores"], "kind": "oracle",
                             "sample": sample, "sweep_gbs": sum(r["sweep_gbs"] for r in results) / len(results)},
            "e2e": {"value": tf, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def summarize_launches(path: str) -> None:
    """Per-kernel launches, total device time and share from an ncu launch list
    (``--metrics gpu__time_duration.sum --csv --log-file``)."""
    import csv
    import io
    text = Path(path).read_text()
    start = text.find('"ID"')
    rows = list(csv.DictReader(io.StringIO(text[start:])))
    tags = {"<1, 1, 1>": "wgrad", "<0, 0, 0>": "fprop", "<0, 1, 0>": "dgrad",
            "<true, true, 1>": "wgrad", "<false, false, 0>": "fprop", "<false, true, 0>": "dgrad"}
    tot: dict = {}
    for r in rows:
        if r.get("Metric Name") != "gpu__time_duration.sum":
            continue
        name = r["Kernel Name"]
        key = name.split("(")[0].replace("<unnamed>::", "").strip()
        if "gemm_bf16" in key and "<" in key:   # name the GEMM by its operand majorness
            base, targs = key.split("<", 1)
            first3 = "<" + ", ".join(a.strip() for a in targs.rstrip(">").split(",")[:3]) + ">"
            key = f"{base.replace('void ', '').strip()} [{tags.get(first3, first3)}]"
        scale = {"ns": 1e-3, "us": 1.0, "usecond": 1.0, "ms": 1e3, "nsecond": 1e-3}.get(r["Metric Unit"], 1e-3)
        v = tot.setdefault(key, [0, 0.0])
        v[0] += 1
        v[1] += float(r["Metric Value"].replace(",", "")) * scale
    total = sum(v[1] for v in tot.values())
    print(f"| kernel | launches | total us | share |\n|---|---:|---:|---:|")
    for k, (n, t) in sorted(tot.items(), key=lambda x: -x[1][1]):
        print(f"| {k} | {n} | {t:.1f} | {100 * t / total:.1f}% |")


def main():
    args = parse()
    if args.summarize_launches:
        return summarize_launches(args.summarize_launches)
    if args.source_hash:
        return print(gemm_source_hash())
    ws, rank, local, pg = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    import torch
    import param_buffers_gb300 as gtp
    from param_buffers_gb300 import workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk, pk_kind = peaks()
    if args.only:
        return run_only(args, torch, gtp, W, dev)
    # The standalone sweeps on the 7B-style buffer run first (13 bf16 + 13 MXFP8 launches),
    # so that a profiler can skip them and capture the layer steps alone.
    sweep = time_sweep_7b(torch, gtp, W, dev)
    sweep["frac"] = sweep["gbs"] / pk["hbm_gbs"]
    sweep["mxfp8"]["frac"] = sweep["mxfp8"]["gbs"] / pk["hbm_gbs"]
    sweep["grad_norm"]["frac"] = sweep["grad_norm"]["gbs"] / pk["hbm_gbs"]
    sweep["bf16_grad"]["frac"] = sweep["bf16_grad"]["gbs"] / pk["hbm_gbs"]
    sweep["rs_local_sum"]["frac"] = sweep["rs_local_sum"]["gbs"] / pk["hbm_gbs"]
    sweep["peak_gbs"] = pk["hbm_gbs"]
    step = LayerStep(dev, seed_offset=rank, schedule=args.schedule)
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    clocks = clock_sampler(local)
    time.sleep(0.6)                         # let the sampler start before the timed region
    s_ev = torch.cuda.Event(enable_timing=True)
    e_ev = torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    s_ev.record()
    for _ in range(args.steps):             # the timed region: nothing but the steps
        step.run()
    host_enqueue_ms = (time.time() - t0) * 1e3 / args.steps
    e_ev.record()
    torch.cuda.synchronize()
    t1 = time.time()
    if pg:
        pg.barrier()
    # A second timed pass of the same steps with CUDA events around every launch gives
    # the per-kernel table and the roofline (events between launches keep kernels from
    # overlapping, so this pass is slightly slower than the one above).
    timer = KernelTimer(torch)
    k_steps = args.steps
    side, step.side = step.side, None       # one stream here: a launch's events bracket it alone
    sched = step.schedule
    if sched == "separate":
        step.schedule = "one-stream"
    # the same idle start as the timed region (it began after the sampler's 0.6 s), so that
    # both passes start from the same power state rather than this one inheriting the
    # power cap the timed region ran into
    torch.cuda.synchronize()
    time.sleep(0.6)
    t2 = time.time()
    for _ in range(k_steps):
        step.run(timer)
    torch.cuda.synchronize()
    t3 = time.time()
    step.side = side
    step.schedule = sched
    clocks.stop()
    ms_total = reduce_max(pg, s_ev.elapsed_time(e_ev))
    ms_step = ms_total / args.steps
    value = step.flops * ws / (ms_step / 1e3) / 1e12
    totals = timer.totals()

    kinds = {}
    for kind, (ms, n) in totals.items():
        k = kind[0] if isinstance(kind, tuple) else kind
        kinds.setdefault(k, [0.0, 0])
        kinds[k][0] += ms
        kinds[k][1] += n
    gemm_flops = {}
    for kind, (ms, n) in totals.items():
        if isinstance(kind, tuple):
            gemm_flops[kind[0]] = gemm_flops.get(kind[0], 0) + step.kind_flops[kind] * n
    per_kernel = {k: {"ms_total": ms, "launches": n,
                      "tflops": gemm_flops[k] / (ms / 1e3) / 1e12 if k in gemm_flops else None}
                  for k, (ms, n) in kinds.items()}
    per_kernel["adam"]["gbs"] = SWEEP_BYTES_PER_ELEM * step.numel * args.steps / (kinds["adam"][0] / 1e3) / 1e9
    per_kernel["mxfp8"]["tflops"] = step.mx_flops * args.steps / (kinds["mxfp8"][0] / 1e3) / 1e12
    per_kernel["gradnorm"]["gbs"] = 4 * step.numel * args.steps / (kinds["gradnorm"][0] / 1e3) / 1e9
    # quantize: read fp32 masters (4 B) or bf16 X (2 B), write 1 + 1/32 B per element
    q_bytes = sum(l.N * l.K * (4 + 1 + 1 / 32) for l in step.mx_lins) + step.M * step.fc1.K * (2 + 1 + 1 / 32)
    per_kernel["quant"]["gbs"] = q_bytes * args.steps / (kinds["quant"][0] / 1e3) / 1e9
    for kind, (ms, n) in totals.items():
        if isinstance(kind, tuple):
            per_kernel[f"{kind[0]}.{kind[1]}"] = {"ms_per_launch": ms / n,
                                                  "tflops": step.kind_flops[kind] * n / (ms / 1e3) / 1e12}
    # the dominant kernel: the (GEMM, linear) launch shape with the largest device time
    dom_kind, (dom_ms, dom_n) = max(((k, v) for k, v in totals.items() if isinstance(k, tuple)),
                                    key=lambda kv: kv[1][0])
    dims = {l.name: l for l in step.lins}
    burst = pk["bf16_tflops"]
    sustained = pk.get("bf16_tflops_sustained", burst)
    ach = step.kind_flops[dom_kind] * dom_n / (dom_ms / 1e3) / 1e12
    traffic = traffic_from_profiles(f"{dom_kind[0]}.{dom_kind[1]}")
    # the library runs the CTA-pair kernel whenever the output has more than 128 rows
    kname = ("gemm_bf16_kernel" if os.environ.get("GTP_GEMM_VARIANT") == "single" or step.M <= 128
             else "gemm_bf16_group_kernel" if dom_kind[0] in ("backward", "overlap") else "gemm_bf16_pair_kernel")
    shape = ", ".join(f"{n}: N={dims[n].N}, K={dims[n].K}" for n in dom_kind[1].split("+"))
    # A timed region well under a second runs at burst clocks: the burst peak is the
    # denominator; the sustained one (a seconds-long power-capped loop) only past a second.
    region_s = t3 - t2
    long_region = region_s >= 1.0
    peak = sustained if long_region else burst
    clk = clocks.summary(t2, t3)
    peak_mhz = (pk.get("clocks_under_load") or {}).get("sm_mhz_median")
    roofline = {"kernel": f"{kname} {dom_kind[0]} {dom_kind[1]} (M={step.M}; {shape})",
                "bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                "traffic": traffic, "share_of_kernel_time": dom_ms / sum(v[0] for v in totals.values()),
                "peak_source": (f"{pk_kind} bf16_tflops_sustained (timed pass {region_s:.2f} s)" if long_region else
                                f"{pk_kind} bf16_tflops burst (timed pass {region_s:.2f} s, under a second)"),
                "frac_vs_burst": ach / burst, "frac_vs_sustained": ach / sustained}
    bpe = sweep_traffic_per_elem()
    roofline["sweep"] = {
        "kernel": f"adam_flat_kernel: fused scale, AdamW, bf16 cast and zero over the 7B-style flat buffer "
                  f"({sweep['numel']:,} elements)",
        "bound": "hbm", "achieved": sweep["gbs"], "peak": pk["hbm_gbs"], "unit": "GB/s",
        "frac": sweep["gbs"] / pk["hbm_gbs"], "algorithmic_bytes": SWEEP_BYTES_PER_ELEM * sweep["numel"],
        "traffic": None if bpe is None else bpe * sweep["numel"],
        "traffic_source": "ncu dram bytes per element on the layer buffer (30.4M elements), times the elements "
                          "of this launch (profiles/traffic_sweep.txt)",
        "peak_source": f"{pk_kind} hbm_gbs (copy)"}
    if peak_mhz and clk.get("sm_mhz"):
        # the sustained peak was taken at peak_mhz; scaled to this pass's median SM clock,
        # and never above the burst peak (the best the GEMM reaches at any clock)
        scaled = min(burst, sustained * clk["sm_mhz"] / peak_mhz)
        roofline["frac_clock_normalised"] = ach / scaled
        roofline["clock_note"] = (f"sustained peak {sustained} TFLOP/s at a median {peak_mhz:.0f} MHz, scaled to "
                                  f"this pass's median {clk['sm_mhz']:.0f} MHz: {scaled:.1f} TFLOP/s, at most "
                                  f"the burst peak")

    shape_clocks = clock_sampler(local, 0.002)
    time.sleep(0.3)
    shapes = time_gemm_shapes(step, torch, pk, shape_clocks)
    roofline["gemm_shapes_frac_burst"] = {k: round(v["frac_burst"], 3) for k, v in shapes["shapes"].items()}
    time.sleep(0.5)   # each table starts from an idle part, as the timed region does
    lowp = time_lowp_gemms(torch, gtp, W, dev, pk, shape_clocks)
    time.sleep(0.5)
    quant = time_quantize(torch, gtp, W, dev, pk, shape_clocks)
    shape_clocks.stop()
    # compact fractions of the other kernels' rooflines, beside the dominant one
    roofline["lowp_frac"] = {k: round(v["frac"], 3) for k, v in lowp.items()}
    roofline["lowp_frac_of_mma_rate"] = {k: round(v["frac_of_mma_rate"], 3) for k, v in lowp.items()}
    roofline["rs_local_sum_frac_hbm"] = round(sweep["rs_local_sum"]["frac"], 3)
    roofline["quantize_frac_hbm"] = {k: round(v["frac"], 3) for k, v in quant.items()}
    e2e = run_e2e(step, torch, args.e2e_steps, pg, ws, args.copy_streams, args.e2e_reps)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        o = oracle_sample(seconds=10.0)
        cpu = {"value": o["tflops"], "unit": "TFLOP/s", "cores": o["cores"], "kind": "oracle", "sample": o["sample"],
               "sweep_gbs": o["sweep_gbs"]}
    launches = step.launches_per_step * args.steps
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": layer_config(W, ws, torch.cuda.get_device_properties(dev).multi_processor_count),
            "roofline": roofline,
            "adamw_sweep": {"workload": "7B-style flat buffer, 1.875e9 params, 31 buckets; the fused sweep, its "
                                        "native-MXFP8 form and the gradient-norm pass over the same buffer",
                            "bytes_per_elem": SWEEP_BYTES_PER_ELEM, **sweep, "unit": "GB/s",
                            "peak_source": f"{pk_kind} hbm_gbs"},
            "lowp_gemms": {"workload": "fc1 shape M 8192, N 8192, K 2048, operands quantized up front, each GEMM "
                                       "alone (batches of 8 back-to-back launches, median of 10)", **lowp},
            "quantize": {"workload": "W_fc1 [8192,2048] and W_fc2 [2048,8192] fp32, X [8192,2048] bf16, each "
                                     "launch on the next source of the three (168 MB, more than L2), batches of "
                                     "three rotations, median of 20; peak = measured HBM copy GB/s", **quant},
            "kernels": per_kernel,
            "gemm_shapes": shapes,
            "e2e": e2e,
            "gpu_launches": launches,
            "host_enqueue_ms_per_step": host_enqueue_ms,
            "schedule": step.schedule,
            "clocks": clocks.summary(t0, t1),
            "kernel_timing_pass": {"steps": k_steps, "note": "per-kernel events; kernels and roofline come from it; "
                                                           "started after the same 0.6 s idle as the timed region",
                                   "clocks": clocks.summary(t2, t3)},
        }
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def batch_ms(torch, launch, n: int, per_batch: int = 10) -> float:
    """ms per launch of n launches, timed in batches of back-to-back launches (CUDA events
    around each batch on the launching stream; the median over batches).  Timing single
    launches between synchronisations would add the host's time to enqueue the call
    (about 10 us through the Python binding) to every figure."""
    ts = []
    done = 0
    while done < n:
        b = min(per_batch, n - done)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for i in range(b):
            launch(done + i)
        e.record()
        e.synchronize()
        ts.append(s.elapsed_time(e) / b)
        done += b
    return sorted(ts)[len(ts) // 2]


def time_gemm_shapes(step, torch, pk, clocks, reps: int = 10) -> dict:
    """Each of the layer's twelve bf16 GEMM launch shapes alone, launched the way the step
    launches them: back to back on one stream (each launch may start its set-up under the
    previous one's tail), one launch per microbatch on that microbatch's inputs (0.3-3 GB
    across the eight, more than L2).  CUDA events around each batch of eight, median over
    `reps` batches; frac against the measured bf16 burst peak (these batches last well
    under a second)."""
    gtp = step.gtp
    burst = pk["bf16_tflops"]
    nmb = len(step.X)
    out = {}
    for lin in step.lins:
        Wv = step.weight(lin)
        calls = {
            "fprop": lambda mb, lin=lin, Wv=Wv: gtp.gtp_linear_fprop(step.X[mb][lin.name], Wv, step.Y[lin.name]),
            "dgrad": lambda mb, lin=lin, Wv=Wv: gtp.gtp_linear_dgrad(step.dY[mb][lin.name], Wv, step.dX[lin.name]),
            "wgrad": lambda mb, lin=lin: gtp.gtp_linear_wgrad_accum(step.dY[mb][lin.name], step.X[mb][lin.name],
                                                                    step.grad, step.offsets[lin.name]),
        }
        calls["backward"] = lambda mb, lin=lin, Wv=Wv: gtp.gtp_linear_backward(
            step.dY[mb][lin.name], step.X[mb][lin.name], Wv, step.dX[lin.name], step.grad, step.offsets[lin.name])
        for kind, fn in calls.items():
            for mb in range(nmb):
                fn(mb)
            torch.cuda.synchronize()
            t0 = time.time()
            ms = batch_ms(torch, lambda i, fn=fn: fn(i % nmb), reps * nmb, per_batch=nmb)
            clk = clocks.summary(t0, time.time())
            tf = step.W.linear_flops(step.M, lin.N, lin.K) * (2 if kind == "backward" else 1) / (ms / 1e3) / 1e12
            out[f"{kind}.{lin.name}"] = {"us_per_launch": ms * 1e3, "tflops": tf, "frac_burst": tf / burst,
                                         "sm_mhz": clk.get("sm_mhz"), "clock_samples": clk.get("samples")}
    torch.cuda.synchronize()
    worst = min(out, key=lambda k: out[k]["frac_burst"])
    return {"workload": "each layer GEMM shape alone: batches of 8 back-to-back launches on the 8 microbatches' "
                        "inputs, median of 10 batches", "peak_tflops": burst,
            "peak_source": "measured bf16_tflops (burst)", "shapes": out,
            "min_frac_burst": out[worst]["frac_burst"], "min_shape": worst}


LOWP_NAMES = ("mxfp8_fprop", "mxfp8_dgrad", "mxfp8_wgrad", "nvfp4_fprop", "mxfp8_fprop_tiled", "nvfp4_fprop_tiled",
              "mxfp8_dgrad_tiled", "mxfp8_wgrad_tiled")


def lowp_gemms(torch, gtp, W, dev) -> dict:
    """The fc1 shape (M 8192, N 8192, K 2048) on the block-scaled paths: MXFP8 fprop, dgrad
    and wgrad-accumulate, and NVFP4 fprop, each MXFP8 GEMM and the NVFP4 forward also with
    tiled scales.  The operands are quantized once up front (the
    optimizer-step and per-forward quantize are timed elsewhere); returns name -> (launch,
    FLOP per launch, peak key)."""
    lin = next(l for l in W.LAYER_LINEARS if l.name == "fc1")
    M, N, K = W.LAYER_M, lin.N, lin.K
    g = W.generator(W.seed_of("mxfp8") + 1, dev)
    X, Wt, dY = W.linear_inputs(M, N, K, g, dev)
    u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device=dev)
    Xq, Xs, Wq, Ws = u8(M, K), u8(M, K // 32), u8(N, K), u8(N, K // 32)
    dYq, dYs, Wtq, Wts = u8(M, N), u8(M, N // 32), u8(K, N), u8(K, N // 32)
    dYtq, dYts, Xtq, Xts = u8(N, M), u8(N, M // 32), u8(K, M), u8(K, M // 32)
    gtp.gtp_mxfp8_quantize_rowwise(X, Xq, Xs)
    gtp.gtp_mxfp8_quantize_rowwise(Wt, Wq, Ws)
    gtp.gtp_mxfp8_quantize_rowwise(dY, dYq, dYs)
    gtp.gtp_mxfp8_quantize_columnwise(Wt, Wtq, Wts)
    gtp.gtp_mxfp8_quantize_columnwise(dY, dYtq, dYts)
    gtp.gtp_mxfp8_quantize_columnwise(X, Xtq, Xts)
    f32 = lambda n: torch.zeros(n, dtype=torch.float32, device=dev)
    Xp, Xps, xa, Wp, Wps, wa = u8(M, K // 2), u8(M, K // 16), f32(1), u8(N, K // 2), u8(N, K // 16), f32(1)
    gtp.gtp_nvfp4_quantize_rowwise(X, Xp, Xps, xa)
    gtp.gtp_nvfp4_quantize_rowwise(Wt, Wp, Wps, wa)
    # the same scales in the tiled layout (the fused tiled quantize writes identical codes)
    tiled = lambda rows, cols: u8(gtp.gtp_sf_tiled_bytes(rows, cols))
    Xst, Wst, Xpst, Wpst = tiled(M, K // 32), tiled(N, K // 32), tiled(M, K // 16), tiled(N, K // 16)
    gtp.gtp_mxfp8_quantize_rowwise_tiled(X, Xq, Xst)
    gtp.gtp_mxfp8_quantize_rowwise_tiled(Wt, Wq, Wst)
    gtp.gtp_nvfp4_quantize_rowwise_tiled(X, Xp, Xpst, xa)
    gtp.gtp_nvfp4_quantize_rowwise_tiled(Wt, Wp, Wpst, wa)
    dYst, Wtst, dYtst, Xtst = tiled(M, N // 32), tiled(K, N // 32), tiled(N, M // 32), tiled(K, M // 32)
    gtp.gtp_mxfp8_quantize_rowwise_tiled(dY, dYq, dYst)
    gtp.gtp_mxfp8_quantize_columnwise_group([(Wt, Wtq, Wtst), (dY, dYtq, dYtst), (X, Xtq, Xtst)])
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    dX = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    mg = f32(N * K)
    fl = W.linear_flops(M, N, K)
    return {
        "mxfp8_fprop": (lambda: gtp.gtp_linear_fprop_mxfp8(Xq, Xs, Wq, Ws, Y), fl, "fp8"),
        "mxfp8_dgrad": (lambda: gtp.gtp_linear_dgrad_mxfp8(dYq, dYs, Wtq, Wts, dX), fl, "fp8"),
        "mxfp8_wgrad": (lambda: gtp.gtp_linear_wgrad_accum_mxfp8(dYtq, dYts, Xtq, Xts, mg, 0), fl, "fp8"),
        "nvfp4_fprop": (lambda: gtp.gtp_linear_fprop_nvfp4(Xp, Xps, xa, Wp, Wps, wa, Y), fl, "fp4"),
        "mxfp8_fprop_tiled": (lambda: gtp.gtp_linear_fprop_mxfp8_tiled(Xq, Xst, Wq, Wst, Y), fl, "fp8"),
        "nvfp4_fprop_tiled": (lambda: gtp.gtp_linear_fprop_nvfp4_tiled(Xp, Xpst, xa, Wp, Wpst, wa, Y), fl, "fp4"),
        "mxfp8_dgrad_tiled": (lambda: gtp.gtp_linear_dgrad_mxfp8_tiled(dYq, dYst, Wtq, Wtst, dX), fl, "fp8"),
        "mxfp8_wgrad_tiled": (lambda: gtp.gtp_linear_wgrad_accum_mxfp8_tiled(dYtq, dYtst, Xtq, Xtst, mg, 0), fl,
                              "fp8"),
    }


def time_lowp_gemms(torch, gtp, W, dev, pk, clocks=None, reps: int = 20) -> dict:
    """Each block-scaled GEMM alone (batches of 8 back-to-back launches, median over 10
    batches), against the measured bf16 burst peak times the nominal dense ratio of its type
    (fp8 4.5 / 2.25 = 2x, fp4 13.5 / 2.25 = 6x PFLOP/s).  `frac_of_mma_rate` divides instead
    by the bf16 peak times the per-cycle rate of the type's MMA measured against bf16's on
    this GPU (back-to-back MMAs on resident operands: 2x fp8, 4x fp4)."""
    fns = lowp_gemms(torch, gtp, W, dev)
    ratio = {"fp8": 2.0, "fp4": 6.0}
    mma_rate = {"fp8": 2.0, "fp4": 4.0}
    out = {}
    for name, (fn, flops, kind) in fns.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        t0 = time.time()
        ms = batch_ms(torch, lambda i: fn(), 4 * reps, per_batch=8)
        clk = clocks.summary(t0, time.time()) if clocks else {}
        peak = pk["bf16_tflops"] * ratio[kind]
        tf = flops / (ms / 1e3) / 1e12
        out[name] = {"ms": ms, "tflops": tf, "peak_tflops": peak, "frac": tf / peak, "sm_mhz": clk.get("sm_mhz"),
                     "peak_source": f"bf16_tflops x {ratio[kind]:g} (nominal {kind} / bf16 dense ratio)",
                     "frac_of_mma_rate": tf / (pk["bf16_tflops"] * mma_rate[kind])}
    del fns
    torch.cuda.empty_cache()
    return out


QUANT_KINDS = ("mxfp8_rowwise", "mxfp8_rowwise_group", "mxfp8_columnwise", "mxfp8_columnwise_group",
               "nvfp4_rowwise")


def quantize_inputs(torch, gtp, W, dev):
    """The quantize passes' sources (W_fc1 [8192, 2048] and W_fc2 [2048, 8192] fp32 masters
    ~N(0, 0.02), X [8192, 2048] bf16 ~N(0, 1)) with their outputs; run(kind, i) quantizes
    source i (the _group kinds: all three sources in one call),
    nbytes(kind, x) is source x's algorithmic bytes (source read once, NVFP4 twice for its
    amax pass, plus codes and scales written)."""
    g = W.generator(W.seed_of("mxfp8"), dev)
    srcs = [W.randn_f32((R, C), 0.02, g, dev) for _, R, C in W.MXFP8_W] + [W.randn_bf16(W.MXFP8_X, 1.0, g, dev)]
    u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device=dev)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    outs = []
    for x in srcs:
        R, C = x.shape
        outs.append({"q": u8(R, C), "s": u8(R, C // 32), "qt": u8(C, R), "st": u8(C, R // 32),
                     "p": u8(R, C // 2), "ps": u8(R, C // 16)})

    def run(kind, i):
        x, o = srcs[i], outs[i]
        if kind == "mxfp8_rowwise":
            gtp.gtp_mxfp8_quantize_rowwise(x, o["q"], o["s"])
        elif kind == "mxfp8_columnwise":
            gtp.gtp_mxfp8_quantize_columnwise(x, o["qt"], o["st"])
        elif kind == "mxfp8_rowwise_group":
            gtp.gtp_mxfp8_quantize_rowwise_group([(y, p["q"], p["s"]) for y, p in zip(srcs, outs)])
        elif kind == "mxfp8_columnwise_group":
            gtp.gtp_mxfp8_quantize_columnwise_group([(y, p["qt"], p["st"]) for y, p in zip(srcs, outs)])
        else:
            gtp.gtp_nvfp4_quantize_rowwise(x, o["p"], o["ps"], amax)

    def nbytes(kind, x):
        el, src = x.numel(), x.element_size()
        if kind == "nvfp4_rowwise":
            return el * (2 * src + 0.5 + 1 / 16)
        return el * (src + 1 + 1 / 32)

    return srcs, run, nbytes


def time_quantize(torch, gtp, W, dev, pk, clocks=None, reps: int = 20) -> dict:
    """The MXFP8 workload's quantize passes alone: W_fc1 [8192, 2048] and W_fc2 [2048, 8192]
    fp32 masters ~N(0, 0.02), X [8192, 2048] bf16 ~N(0, 1), rowwise and columnwise MXFP8 and
    rowwise NVFP4.  Each launch takes the next source in a rotation over the three (168 MB
    of sources, more than L2), timed in batches of three rotations, against the measured
    HBM copy bandwidth; bytes are algorithmic: source read once (NVFP4: twice, amax pass
    and quantize pass) plus codes and scales written.  The _group kinds quantize the
    three sources in one launch (the rotation's bytes a launch)."""
    srcs, run, nbytes = quantize_inputs(torch, gtp, W, dev)

    out = {}
    for kind in QUANT_KINDS:
        for i in range(3):
            run(kind, i)
        torch.cuda.synchronize()
        t0 = time.time()
        ms = batch_ms(torch, lambda t: run(kind, t % 3), 9 * reps, per_batch=9)  # 3 rotations a batch
        clk = clocks.summary(t0, time.time()) if clocks else {}
        rotation = sum(nbytes(kind, x) for x in srcs)
        gbs = rotation / (1 if kind.endswith("_group") else 3) / (ms / 1e3) / 1e9
        out[kind] = {"us_per_launch": ms * 1e3, "gbs": gbs, "frac": gbs / pk["hbm_gbs"], "sm_mhz": clk.get("sm_mhz")}
    del srcs, run
    torch.cuda.empty_cache()
    return out


def run_only(args, torch, gtp, W, dev):
    """One kernel of the step on one shape, for profilers: warmup + steps launches."""
    if args.only in LOWP_NAMES:
        fn0, flops, _ = lowp_gemms(torch, gtp, W, dev)[args.only]
        fn, work, unit = (lambda t: fn0()), flops / 1e12, "TFLOP/s"
        args.linear = "fc1"
    elif args.only.startswith("quantize_"):
        kind = args.only[len("quantize_"):]
        srcs, run, nbytes = quantize_inputs(torch, gtp, W, dev)
        fn = lambda t: run(kind, t % 3)   # rotates W_fc1, W_fc2, X (a group: all three a launch)
        work, unit = sum(nbytes(kind, x) for x in srcs) / (1 if kind.endswith("_group") else 3) / 1e9, "GB/s"
        args.linear = None
    lin = next((l for l in W.LAYER_LINEARS if l.name == args.linear), None)
    g = W.generator(W.seed_of("layer"), dev)
    if args.only in LOWP_NAMES or args.only.startswith("quantize_"):
        pass
    elif args.only == "overlap":
        nb, nf = args.linear.split("+")
        lb = next(l for l in W.LAYER_LINEARS if l.name == nb)
        lf = next(l for l in W.LAYER_LINEARS if l.name == nf)
        M = W.LAYER_M
        Xb, Wb, dYb = W.linear_inputs(M, lb.N, lb.K, g, dev)
        Xf, Wf, _ = W.linear_inputs(M, lf.N, lf.K, g, dev)
        dX = torch.empty(M, lb.K, dtype=torch.bfloat16, device=dev)
        Yf = torch.empty(M, lf.N, dtype=torch.bfloat16, device=dev)
        mg = torch.zeros(lb.N * lb.K, device=dev)
        descs = [gtp.gemm_desc("dgrad", dYb, Wb, dX), gtp.gemm_desc("wgrad", dYb, Xb, mg),
                 gtp.gemm_desc("fprop", Xf, Wf, Yf)]
        fn = lambda t: gtp.gtp_linear_grouped(descs)
        work, unit = (2 * W.linear_flops(M, lb.N, lb.K) + W.linear_flops(M, lf.N, lf.K)) / 1e12, "TFLOP/s"
    elif args.only == "rs_local_sum":
        P, n = 64, 1_000_000       # the 7B buffer's bucket shard at dp 64
        sets = [W.randn_bf16((P, n), 1e-3, g, dev) for _ in range(3)]
        outs = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(3)]
        fn = lambda t: gtp.gtp_rs_local_sum(sets[t % 3], outs[t % 3])
        work, unit = (P + 1) * 2 * n / 1e9, "GB/s"
    elif args.only in ("adam", "adam_mx", "gradnorm"):
        n = args.sweep_numel
        grad, master, m, v, param = W.buffer_state(n, g, dev)
        one = [{"offset": 0, "numel": n}]
        if args.only == "adam":
            fn = lambda t: gtp.gtp_adam_step_flat(grad, master, m, v, param, one, [0.5], gtp.AdamHparams(), step=t)
            work = SWEEP_BYTES_PER_ELEM * n / 1e9
        elif args.only == "adam_mx":
            q = torch.empty(n, dtype=torch.uint8, device=dev)
            sc = torch.empty(n // 32, dtype=torch.uint8, device=dev)
            fn = lambda t: gtp.gtp_adam_step_flat_mxfp8(grad, master, m, v, q, sc, one, [0.5], gtp.AdamHparams(),
                                                        step=t)
            work = SWEEP_MX_BYTES_PER_ELEM * n / 1e9
        else:
            ws = torch.empty(max(16, gtp.gtp_grad_norm_workspace_bytes(one)), dtype=torch.uint8, device=dev)
            outs = (torch.empty(1, dtype=torch.float64, device=dev), torch.empty(1, dtype=torch.int32, device=dev),
                    torch.empty(1, device=dev), torch.empty(1, device=dev))
            fn = lambda t: gtp.gtp_grad_norm(grad, one, [0.5], 1.0, ws, *outs)
            work = 4 * n / 1e9
        unit = "GB/s"
    else:
        M = W.LAYER_M
        X, Wt, dY = W.linear_inputs(M, lin.N, lin.K, g, dev)
        Y = torch.empty(M, lin.N, dtype=torch.bfloat16, device=dev)
        dX = torch.empty(M, lin.K, dtype=torch.bfloat16, device=dev)
        mg = torch.zeros(lin.N * lin.K, device=dev)
        fn = {"fprop": lambda t: gtp.gtp_linear_fprop(X, Wt, Y), "dgrad": lambda t: gtp.gtp_linear_dgrad(dY, Wt, dX),
              "wgrad": lambda t: gtp.gtp_linear_wgrad_accum(dY, X, mg, 0),
              "wgrad_det": lambda t: gtp.gtp_linear_wgrad_accum(dY, X, mg, 0, deterministic=True),
              "backward": lambda t: gtp.gtp_linear_backward(dY, X, Wt, dX, mg, 0)}[args.only]
        work, unit = W.linear_flops(M, lin.N, lin.K) * (2 if args.only == "backward" else 1) / 1e12, "TFLOP/s"
    for t in range(args.warmup):
        fn(t + 1)
    torch.cuda.synchronize()
    # the same launch sequence as before batching (warm-up, then `steps` launches), so a
    # profiler's skip / count arguments select the same launches
    ms = batch_ms(torch, lambda t: fn(args.warmup + t + 1), args.steps)
    print(json.dumps({"only": args.only, "linear": args.linear if args.only in ("fprop", "dgrad", "wgrad", "wgrad_det", "backward", "overlap") else None,
                      "ms_per_launch": ms, "value": work / (ms / 1e3), "unit": unit}), flush=True)


def run_e2e(step, torch, steps, pg, ws, copy_streams: int = 2, n_reps: int = 15) -> dict:
    """The same step through the public API with host inputs: each step copies that
    step's activations and upstream gradients from pinned host memory and reads the
    updated bf16 parameters back.  The device inputs are double-buffered: while step i
    computes on one set, the copies of step i + 1 fill the other, microbatch by microbatch
    on their own streams; a microbatch's GEMMs wait only for their own inputs, and a set is
    refilled only after the step that read it (two steps earlier) is done with it."""
    host_X = [{k: t.cpu().pin_memory() for k, t in d.items()} for d in step.X]
    host_dY = [{k: t.cpu().pin_memory() for k, t in d.items()} for d in step.dY]
    out = torch.empty(step.numel, dtype=torch.bfloat16).pin_memory()
    h2d = sum(t.numel() * t.element_size() for d in (*host_X, *host_dY) for t in d.values())
    d2h = out.numel() * out.element_size()
    comp = torch.cuda.current_stream()
    copiers = [torch.cuda.Stream() for _ in range(copy_streams)]
    nmb = len(step.X)
    sets = [(step.X, step.dY),
            ([{k: torch.empty_like(t) for k, t in d.items()} for d in step.X],
             [{k: torch.empty_like(t) for k, t in d.items()} for d in step.dY])]
    ready = [[torch.cuda.Event() for _ in range(nmb)] for _ in sets]
    free = [torch.cuda.Event() for _ in sets]   # the set's last reader (a whole step) is done
    for ev in free:
        ev.record(comp)

    def copy_in(i):
        X, dY = sets[i % 2]
        for mb in range(nmb):
            cs = copiers[mb % len(copiers)]
            cs.wait_event(free[i % 2])
            with torch.cuda.stream(cs):
                for k in X[mb]:
                    X[mb][k].copy_(host_X[mb][k], non_blocking=True)
                for k in dY[mb]:
                    dY[mb][k].copy_(host_dY[mb][k], non_blocking=True)
            ready[i % 2][mb].record(cs)

    def compute(i):
        step.X, step.dY = sets[i % 2]
        waited = set()
        for need, op in step.plan():
            if need is not None and need not in waited:
                for mb in range(need + 1):           # a microbatch's launches wait for its own inputs
                    if mb not in waited:
                        comp.wait_event(ready[i % 2][mb])
                        waited.add(mb)
            op(None)
        free[i % 2].record(comp)
        out.copy_(step.param, non_blocking=True)

    def run(n):
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)  # the next step's inputs flow in while this one computes
            compute(i)

    def copy_ceiling() -> float:
        """ms for one step's inputs on the same streams with no compute (second of two passes)."""
        t = 0.0
        for rep in range(2):  # the first pass warms the copy path up
            torch.cuda.synchronize()
            s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(comp)
            for ev in free:
                ev.record(comp)
            copy_in(0)
            for mb in range(nmb):
                comp.wait_event(ready[0][mb])
            e0.record(comp)
            torch.cuda.synchronize()
            t = s0.elapsed_time(e0)
        return t

    h2d_ms = copy_ceiling()
    run(2)
    torch.cuda.synchronize()
    # The host link is shared with the machine's other jobs: now and then one step's copies
    # stall for 60-160 ms (a continuous run holds the copy-bound rate between stalls).  The
    # loop is timed as many short repetitions, so that most of them fall between stalls, and
    # the median reported, with every repetition and the mean over all of them beside it.
    reps, host_ms = [], 0.0
    for _ in range(n_reps):
        if pg:
            pg.barrier()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        h0 = time.perf_counter()
        run(steps)
        host_ms = (time.perf_counter() - h0) * 1e3 / steps  # the host's enqueue time per step
        e.record()
        torch.cuda.synchronize()
        reps.append(reduce_max(pg, s.elapsed_time(e)) / steps)
    h2d_after_ms = copy_ceiling()
    step.X, step.dY = sets[0]
    ms = sorted(reps)[len(reps) // 2]
    mean_ms = sum(reps) / len(reps)
    return {"value": step.flops * ws / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "repetitions_ms_per_step": reps, "statistic": "median of the repetitions",
            "value_fastest_repetition": step.flops * ws / (min(reps) / 1e3) / 1e12,
            "value_mean_of_repetitions": step.flops * ws / (mean_ms / 1e3) / 1e12,
            "host_enqueue_ms_per_step": host_ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps, "repetitions": n_reps,
            "copy_streams": copy_streams, "h2d_alone_ms": h2d_ms, "h2d_alone_gbs": h2d / h2d_ms / 1e6,
            "h2d_alone_gbs_after": h2d / h2d_after_ms / 1e6,
            "overlap": "double-buffered device inputs: the next step's host-to-device copies overlap this "
                       "step's GEMMs, microbatch by microbatch on their own streams"}


if __name__ == "__main__":
    main()
