"""Python binding of libgtp.so: the GB300 hot path of a tensor-parallel linear layer
and its flat param/grad buffer.

Each function has the name of the C entry point it calls (``include/gtp.h``) and does
argument marshalling only: it takes torch tensors for device memory, passes their
pointers, sizes and the current CUDA stream, and raises ``GtpError`` on a non-OK
status.  Every step of the path runs in the library's own kernels; there is no
fallback.  ``gtp_buffer_layout`` is host-only and needs no GPU.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import Sequence

from . import abi

__all__ = [
    "GtpError", "ParamDesc", "LayoutConfig", "AdamHparams", "Layout", "lib",
    "gtp_linear_fprop", "gtp_linear_dgrad", "gtp_linear_wgrad_accum", "gtp_linear_backward", "gtp_linear_grouped",
    "GemmDesc", "gemm_desc", "gtp_buffer_layout",
    "gtp_buffer_zero", "gtp_bucket_scale", "gtp_adam_step_flat", "gtp_adam_step_flat_mxfp8", "gtp_grad_norm",
    "gtp_grad_norm_workspace_bytes", "gtp_grad_norm_noalloc", "gtp_shard_param_ranges",
    "gtp_mxfp8_quantize_rowwise", "gtp_mxfp8_quantize_columnwise", "gtp_mxfp8_quantize_columnwise_group",
    "gtp_mxfp8_quantize_columnwise_tiled", "gtp_linear_dgrad_mxfp8_tiled", "gtp_linear_wgrad_accum_mxfp8_tiled",
    "gtp_mxfp8_quantize_rowwise_group", "gtp_rs_local_sum",
    "gtp_linear_fprop_mxfp8",
    "gtp_linear_dgrad_mxfp8", "gtp_linear_wgrad_accum_mxfp8", "gtp_nvfp4_quantize_rowwise",
    "gtp_linear_fprop_nvfp4", "gtp_sf_tiled_bytes", "gtp_sf_tile", "gtp_mxfp8_quantize_rowwise_tiled",
    "gtp_nvfp4_quantize_rowwise_tiled", "gtp_linear_fprop_mxfp8_tiled", "gtp_linear_fprop_nvfp4_tiled",
    "gtp_wait_timeouts", "gtp_selftest_wait_timeout",
]


class GtpError(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        super().__init__(f"{fn}: {abi.STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def lib() -> C.CDLL:
    return abi.load()


def _check(status: int, fn: str) -> None:
    if status != abi.GTP_OK:
        raise GtpError(status, fn, (lib().gtp_last_error() or b"").decode(errors="replace"))


def _stream(stream) -> int:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _require(t, dtype, name: str, ndim: int | None = None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


# ----------------------------------------------------------------------------- GEMMs

def gtp_linear_fprop(X, W, Y, stream=None) -> None:
    """Y[M,N] = X[M,K] W[N,K]^T (bf16 in and out, fp32 accumulation)."""
    import torch
    for t, n in ((X, "X"), (W, "W"), (Y, "Y")):
        _require(t, torch.bfloat16, n, 2)
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K or tuple(Y.shape) != (M, N):
        raise ValueError("shape mismatch: X [M,K], W [N,K], Y [M,N]")
    _check(lib().gtp_linear_fprop(_ptr(X), _ptr(W), _ptr(Y), M, N, K, abi.GTP_BF16, _stream(stream)),
           "gtp_linear_fprop")


def gtp_linear_dgrad(dY, W, dX, stream=None) -> None:
    """dX[M,K] = dY[M,N] W[N,K]."""
    import torch
    for t, n in ((dY, "dY"), (W, "W"), (dX, "dX")):
        _require(t, torch.bfloat16, n, 2)
    M, N = dY.shape
    K = W.shape[1]
    if W.shape[0] != N or tuple(dX.shape) != (M, K):
        raise ValueError("shape mismatch: dY [M,N], W [N,K], dX [M,K]")
    _check(lib().gtp_linear_dgrad(_ptr(dY), _ptr(W), _ptr(dX), M, N, K, abi.GTP_BF16, _stream(stream)),
           "gtp_linear_dgrad")


def gtp_linear_wgrad_accum(dY, X, grad_data, grad_offset: int, stream=None, deterministic: bool = False) -> None:
    """grad_data[grad_offset : grad_offset + N*K].view(N, K) += dY[M,N]^T X[M,K], accumulated in fp32.
    deterministic=True calls gtp_linear_wgrad_accum_deterministic (bit-reproducible); a bfloat16
    grad_data calls gtp_linear_wgrad_accum_bf16."""
    import torch
    _require(dY, torch.bfloat16, "dY", 2)
    _require(X, torch.bfloat16, "X", 2)
    if grad_data.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"grad_data must be float32 or bfloat16, got {grad_data.dtype}")
    _require(grad_data, grad_data.dtype, "grad_data")
    M, N = dY.shape
    if X.shape[0] != M:
        raise ValueError("dY and X must have the same number of rows M")
    K = X.shape[1]
    if grad_data.dtype == torch.bfloat16:   # a bf16 grad buffer: always the unsplit accumulate
        name = "gtp_linear_wgrad_accum_bf16"
    else:
        name = "gtp_linear_wgrad_accum_deterministic" if deterministic else "gtp_linear_wgrad_accum"
    _check(getattr(lib(), name)(_ptr(dY), _ptr(X), _ptr(grad_data), int(grad_offset),
                                grad_data.numel(), M, N, K, abi.GTP_BF16, _stream(stream)), name)


def gtp_linear_backward(dY, X, W, dX, grad_data, grad_offset: int, stream=None, deterministic: bool = False) -> None:
    """One launch for a linear's backward: dX[M,K] = dY[M,N] W[N,K] and
    grad_data[grad_offset : grad_offset + N*K].view(N, K) += dY^T X[M,K] (fp32)."""
    import torch
    for t, n in ((dY, "dY"), (X, "X"), (W, "W"), (dX, "dX")):
        _require(t, torch.bfloat16, n, 2)
    _require(grad_data, torch.float32, "grad_data")
    M, N = dY.shape
    K = W.shape[1]
    if W.shape[0] != N or tuple(X.shape) != (M, K) or tuple(dX.shape) != (M, K):
        raise ValueError("shape mismatch: dY [M,N], X [M,K], W [N,K], dX [M,K]")
    _check(lib().gtp_linear_backward(_ptr(dY), _ptr(X), _ptr(W), _ptr(dX), _ptr(grad_data), int(grad_offset),
                                     grad_data.numel(), M, N, K, abi.GTP_BF16,
                                     abi.GTP_GEMM_DETERMINISTIC if deterministic else 0, _stream(stream)),
           "gtp_linear_backward")


@dataclass(frozen=True)
class GemmDesc:
    """One product of gtp_linear_grouped: the C descriptor and the tensors it points into
    (held here so that they stay alive until the call)."""
    c: object
    tensors: tuple


def gemm_desc(kind: str, a, b, out, grad_offset: int = 0) -> GemmDesc:
    """A product for gtp_linear_grouped.  kind: "fprop" (a = X, b = W, out = Y),
    "dgrad" (a = dY, b = W, out = dX) or "wgrad" (a = dY, b = X, out = grad_data: the
    flat fp32 or bf16 grad buffer, grad_offset the first element of the view)."""
    import torch
    for t, n in ((a, "a"), (b, "b")):
        _require(t, torch.bfloat16, n, 2)
    if kind == "fprop":
        _require(out, torch.bfloat16, "out", 2)
        (M, K), N = a.shape, b.shape[0]
        if b.shape[1] != K or tuple(out.shape) != (M, N):
            raise ValueError("shape mismatch: X [M,K], W [N,K], Y [M,N]")
        code, total = abi.GTP_GEMM_FPROP, 0
    elif kind == "dgrad":
        _require(out, torch.bfloat16, "out", 2)
        (M, N), K = a.shape, b.shape[1]
        if b.shape[0] != N or tuple(out.shape) != (M, K):
            raise ValueError("shape mismatch: dY [M,N], W [N,K], dX [M,K]")
        code, total = abi.GTP_GEMM_DGRAD, 0
    elif kind == "wgrad":
        if out.dtype not in (torch.float32, torch.bfloat16):
            raise TypeError(f"out: expected a float32 or bfloat16 grad buffer, got {out.dtype}")
        _require(out, out.dtype, "out")
        (M, N), K = a.shape, b.shape[1]
        if b.shape[0] != M:
            raise ValueError("dY and X must have the same number of rows M")
        code, total = abi.GTP_GEMM_WGRAD_ACCUM, out.numel()
        grad_dtype = abi.GTP_BF16 if out.dtype == torch.bfloat16 else abi.GTP_F32
    else:
        raise ValueError(f"unknown product kind {kind!r}")
    if kind != "wgrad":
        grad_dtype = abi.GTP_F32
    return GemmDesc(abi.gtp_gemm_desc(code, abi.GTP_BF16, _ptr(a), _ptr(b), _ptr(out), M, N, K, int(grad_offset),
                                      total, grad_dtype, 0), (a, b, out))


def gtp_linear_grouped(descs: Sequence[GemmDesc], stream=None, deterministic: bool = False) -> None:
    """Runs up to four independent products (gemm_desc(...) each) in one launch."""
    arr = (abi.gtp_gemm_desc * max(len(descs), 1))(*[d.c for d in descs])
    _check(lib().gtp_linear_grouped(arr, len(descs), abi.GTP_GEMM_DETERMINISTIC if deterministic else 0,
                                    _stream(stream)), "gtp_linear_grouped")


# ----------------------------------------------------------------------------- layout

_DTYPES = {"fp32": abi.GTP_F32, "bf16": abi.GTP_BF16, "fp16": abi.GTP_F16, "uint8": abi.GTP_U8}
_DTYPE_NAMES = {v: k for k, v in _DTYPES.items()}


@dataclass(frozen=True)
class ParamDesc:
    numel: int
    dtype: str = "bf16"
    quantized_storage: bool = False
    is_expert_parallel: bool = False
    is_layer_wise: bool = False
    is_shared_embedding: bool = False


@dataclass(frozen=True)
class LayoutConfig:
    bucket_size: int | None = None
    dp_size: int = 1
    use_distributed_optimizer: bool = True
    pad_buckets_for_high_nccl_busbw: bool = False
    grad_reduce_in_fp32: bool = True


@dataclass
class Layout:
    index: list        # per param: dict(start, end, start_in_bucket, end_in_bucket, bucket_id, buffer_id)
    buffers: list      # dict(numel, param_dtype, grad_dtype, is_expert_parallel, is_layer_wise, first_bucket, num_buckets)
    buckets: list      # dict(offset, numel_unpadded, numel, buffer_id, num_params)
    c_buckets: object  # the ctypes gtp_bucket_desc array, ready for the sweep entry points


def _struct_dict(s) -> dict:
    return {name: getattr(s, name) for name, _ in s._fields_}


def gtp_buffer_layout(params: Sequence[ParamDesc], cfg: LayoutConfig) -> Layout:
    """Host-only layout of the flat buffers (params in MODEL order)."""
    n = len(params)
    arr = (abi.gtp_param_desc * max(n, 1))()
    for i, p in enumerate(params):
        arr[i] = abi.gtp_param_desc(int(p.numel), _DTYPES[p.dtype], int(p.quantized_storage),
                                    int(p.is_expert_parallel), int(p.is_layer_wise),
                                    int(p.is_shared_embedding), 0)
    c = abi.gtp_layout_config(int(cfg.bucket_size or 0), int(cfg.dp_size), int(cfg.use_distributed_optimizer),
                              int(cfg.pad_buckets_for_high_nccl_busbw), int(cfg.grad_reduce_in_fp32))
    nbuf, nbkt = C.c_int32(0), C.c_int32(0)
    L = lib()
    _check(L.gtp_buffer_layout(arr, n, C.byref(c), None, None, C.byref(nbuf), None, C.byref(nbkt)),
           "gtp_buffer_layout")
    idx = (abi.gtp_param_index * max(n, 1))()
    bufs = (abi.gtp_buffer_desc * max(nbuf.value, 1))()
    bkts = (abi.gtp_bucket_desc * max(nbkt.value, 1))()
    _check(L.gtp_buffer_layout(arr, n, C.byref(c), idx, bufs, C.byref(nbuf), bkts, C.byref(nbkt)),
           "gtp_buffer_layout")
    buffers = []
    for i in range(nbuf.value):
        d = _struct_dict(bufs[i])
        d["param_dtype"] = _DTYPE_NAMES[d["param_dtype"]]
        d["grad_dtype"] = _DTYPE_NAMES[d["grad_dtype"]]
        buffers.append(d)
    c_buckets = (abi.gtp_bucket_desc * nbkt.value)(*[bkts[i] for i in range(nbkt.value)])
    return Layout(index=[_struct_dict(idx[i]) for i in range(n)], buffers=buffers,
                  buckets=[_struct_dict(bkts[i]) for i in range(nbkt.value)], c_buckets=c_buckets)


def gtp_shard_param_ranges(layout: Layout, buffer_id: int, dp_size: int, dp_rank: int) -> list:
    """Host-only range map of one dp rank (dicts with the fields of gtp_shard_range)."""
    n = len(layout.index)
    idx = (abi.gtp_param_index * max(n, 1))()
    for i, d in enumerate(layout.index):
        idx[i] = abi.gtp_param_index(d["start"], d["end"], d["start_in_bucket"], d["end_in_bucket"], d["bucket_id"],
                                     d["buffer_id"])
    bk = layout.c_buckets
    cnt = C.c_int32(0)
    L = lib()
    _check(L.gtp_shard_param_ranges(idx, n, bk, len(bk), buffer_id, dp_size, dp_rank, None, C.byref(cnt)),
           "gtp_shard_param_ranges")
    out = (abi.gtp_shard_range * max(cnt.value, 1))()
    _check(L.gtp_shard_param_ranges(idx, n, bk, len(bk), buffer_id, dp_size, dp_rank, out, C.byref(cnt)),
           "gtp_shard_param_ranges")
    return [_struct_dict(out[i]) for i in range(cnt.value)]


def bucket_array(buckets: Sequence[dict]):
    """A ctypes gtp_bucket_desc array from dicts with offset / numel (other fields optional)."""
    arr = (abi.gtp_bucket_desc * max(len(buckets), 1))()
    for i, b in enumerate(buckets):
        arr[i] = abi.gtp_bucket_desc(int(b["offset"]), int(b.get("numel_unpadded", b["numel"])),
                                     int(b["numel"]), int(b.get("buffer_id", 0)), int(b.get("num_params", 0)))
    return arr


def _factor_array(factors: Sequence[float]):
    return (C.c_float * max(len(factors), 1))(*[float(f) for f in factors])


def _bucket_args(buckets, factors: Sequence[float]):
    """(ctypes bucket array, bucket count) with one factor per bucket: the C side reads
    n_buckets entries of both host arrays, so a short list must not reach it."""
    if isinstance(buckets, (list, tuple)):
        n = len(buckets)
        arr = bucket_array(buckets)
    else:
        arr = buckets
        n = len(arr)
    if len(factors) != n:
        raise ValueError(f"{len(factors)} factors for {n} buckets: one factor per bucket is needed")
    return arr, n


# ----------------------------------------------------------------------------- sweep

def gtp_buffer_zero(t, stream=None) -> None:
    """t[:] = 0 for a contiguous fp32 / bf16 / fp16 / uint8 tensor."""
    import torch
    dt = {torch.float32: abi.GTP_F32, torch.bfloat16: abi.GTP_BF16, torch.float16: abi.GTP_F16,
          torch.uint8: abi.GTP_U8}.get(t.dtype)
    if dt is None:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    _check(lib().gtp_buffer_zero(_ptr(t), dt, t.numel(), _stream(stream)), "gtp_buffer_zero")


def gtp_bucket_scale(grad_data, buckets, factors: Sequence[float], stream=None) -> None:
    """grad_data[b.offset : b.offset + b.numel] *= factors[b] (fp32, in place)."""
    import torch
    _require(grad_data, torch.float32, "grad_data")
    arr, nb = _bucket_args(buckets, factors)
    _check(lib().gtp_bucket_scale(_ptr(grad_data), grad_data.numel(), arr if nb else None,
                                  _factor_array(factors) if nb else None, nb, _stream(stream)),
           "gtp_bucket_scale")


@dataclass(frozen=True)
class AdamHparams:
    lr: float = 3e-4
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    zero_grad_after: bool = True


def gtp_grad_norm_workspace_bytes(buckets) -> int:
    arr = buckets if not isinstance(buckets, (list, tuple)) else bucket_array(buckets)
    return int(lib().gtp_grad_norm_workspace_bytes(arr, len(arr)))


def gtp_grad_norm(grad_data, buckets, factors: Sequence[float], max_norm: float, workspace, sumsq, nonfinite,
                  total_norm, clip_coef, stream=None) -> None:
    """Per-bucket sums of squares (fp64) and non-finite counts (int32 tensor read as uint32) of
    the scaled gradient, the total norm and the clip coefficient (fp32 scalars), all on the device."""
    import torch
    _require(grad_data, torch.float32, "grad_data")
    _require(sumsq, torch.float64, "sumsq")
    _require(nonfinite, torch.int32, "nonfinite")
    _require(total_norm, torch.float32, "total_norm")
    _require(clip_coef, torch.float32, "clip_coef")
    arr, nb = _bucket_args(buckets, factors)
    if sumsq.numel() < nb or nonfinite.numel() < nb:
        raise ValueError("sumsq and nonfinite need one entry per bucket")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().gtp_grad_norm(_ptr(grad_data), grad_data.numel(), arr, _factor_array(factors), nb, float(max_norm),
                               _ptr(workspace), ws_bytes, _ptr(sumsq), _ptr(nonfinite), _ptr(total_norm),
                               _ptr(clip_coef), _stream(stream)),
           "gtp_grad_norm")


def gtp_adam_step_flat(grad_data, master, exp_avg, exp_avg_sq, param_data, buckets, factors: Sequence[float],
                       h: AdamHparams, step: int, stream=None, grad_scale=None) -> None:
    """The fused scale -> AdamW -> bf16 cast -> zero-grad sweep over the flat buffer.
    grad_scale: optional one-element float32 device tensor (the clip coefficient).  A
    bfloat16 grad_data (grad_reduce_in_fp32 off) calls gtp_adam_step_flat_bf16_grad."""
    import torch
    n = grad_data.numel()
    bf16_grad = isinstance(grad_data, torch.Tensor) and grad_data.dtype == torch.bfloat16
    for t, name in ((grad_data, "grad_data"), (master, "master"), (exp_avg, "exp_avg"), (exp_avg_sq, "exp_avg_sq")):
        _require(t, torch.bfloat16 if (bf16_grad and name == "grad_data") else torch.float32, name)
        if t.numel() != n:
            raise ValueError(f"{name} must have {n} elements")
    _require(param_data, torch.bfloat16, "param_data")
    if param_data.numel() != n:
        raise ValueError(f"param_data must have {n} elements")
    arr, nb = _bucket_args(buckets, factors)
    if grad_scale is not None:
        _require(grad_scale, torch.float32, "grad_scale")
    hp = abi.gtp_adam_hparams(h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, int(h.zero_grad_after), int(step),
                              _ptr(grad_scale) or None)
    name = "gtp_adam_step_flat_bf16_grad" if bf16_grad else "gtp_adam_step_flat"
    _check(getattr(lib(), name)(_ptr(grad_data), _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq),
                                _ptr(param_data), n, arr if nb else None,
                                _factor_array(factors) if nb else None, nb, C.byref(hp), _stream(stream)), name)


def gtp_adam_step_flat_mxfp8(grad_data, master, exp_avg, exp_avg_sq, param_e4m3, param_e8m0, buckets,
                             factors: Sequence[float], h: AdamHparams, step: int, stream=None, grad_scale=None) -> None:
    """The fused sweep for a buffer of native MXFP8 parameters: param_e4m3 [numel] and
    param_e8m0 [numel/32] (uint8) receive the MX blocks of the updated master."""
    import torch
    n = grad_data.numel()
    for t, name in ((grad_data, "grad_data"), (master, "master"), (exp_avg, "exp_avg"), (exp_avg_sq, "exp_avg_sq")):
        _require(t, torch.float32, name)
        if t.numel() != n:
            raise ValueError(f"{name} must have {n} elements")
    _require(param_e4m3, torch.uint8, "param_e4m3")
    _require(param_e8m0, torch.uint8, "param_e8m0")
    if param_e4m3.numel() != n or param_e8m0.numel() != n // 32:
        raise ValueError(f"param_e4m3 must have {n} elements and param_e8m0 {n // 32}")
    arr, nb = _bucket_args(buckets, factors)
    if grad_scale is not None:
        _require(grad_scale, torch.float32, "grad_scale")
    hp = abi.gtp_adam_hparams(h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, int(h.zero_grad_after), int(step),
                              _ptr(grad_scale) or None)
    _check(lib().gtp_adam_step_flat_mxfp8(_ptr(grad_data), _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq),
                                          _ptr(param_e4m3), _ptr(param_e8m0), n, arr if nb else None,
                                          _factor_array(factors) if nb else None, nb, C.byref(hp),
                                          _stream(stream)),
           "gtp_adam_step_flat_mxfp8")


# ----------------------------------------------------------------------------- MXFP8

def gtp_mxfp8_quantize_rowwise(src, e4m3, e8m0, stream=None) -> None:
    """src[R,C] (fp32 or bf16) -> e4m3[R,C] (uint8), e8m0[R,C/32] (uint8)."""
    import torch
    dt = {torch.float32: abi.GTP_F32, torch.bfloat16: abi.GTP_BF16}.get(src.dtype)
    if dt is None:
        raise TypeError("src must be float32 or bfloat16")
    _require(src, src.dtype, "src", 2)
    R, Cc = src.shape
    _require(e4m3, torch.uint8, "e4m3", 2)
    _require(e8m0, torch.uint8, "e8m0", 2)
    if tuple(e4m3.shape) != (R, Cc) or tuple(e8m0.shape) != (R, Cc // 32):
        raise ValueError("e4m3 must be [R,C] and e8m0 [R,C/32]")
    _check(lib().gtp_mxfp8_quantize_rowwise(_ptr(src), dt, R, Cc, _ptr(e4m3), _ptr(e8m0), _stream(stream)),
           "gtp_mxfp8_quantize_rowwise")


def gtp_mxfp8_quantize_rowwise_group(views: Sequence, stream=None) -> None:
    """Up to eight (src, e4m3, e8m0) triples, each as gtp_mxfp8_quantize_rowwise (a 2-D
    e8m0 [R,C/32]) or gtp_mxfp8_quantize_rowwise_tiled (a 1-D tiled e8m0), in one launch."""
    import torch
    descs = []
    for src, q, s in views:
        dt = {torch.float32: abi.GTP_F32, torch.bfloat16: abi.GTP_BF16}.get(src.dtype)
        if dt is None:
            raise TypeError("src must be float32 or bfloat16")
        _require(src, src.dtype, "src", 2)
        R, Cc = src.shape
        _require(q, torch.uint8, "e4m3", 2)
        if tuple(q.shape) != (R, Cc):
            raise ValueError("e4m3 must be [R,C]")
        tiled = s.dim() == 1
        if tiled:
            _require_tiled(s, R, Cc // 32, "e8m0_tiled")
        else:
            _require(s, torch.uint8, "e8m0", 2)
            if tuple(s.shape) != (R, Cc // 32):
                raise ValueError("e8m0 must be [R,C/32]")
        descs.append(abi.gtp_mx_row_desc(_ptr(src), _ptr(q), _ptr(s), R, Cc, dt, int(tiled)))
    arr = (abi.gtp_mx_row_desc * max(len(descs), 1))(*descs)
    _check(lib().gtp_mxfp8_quantize_rowwise_group(arr, len(descs), _stream(stream)),
           "gtp_mxfp8_quantize_rowwise_group")


def gtp_linear_fprop_mxfp8(Xq, Xs, Wq, Ws, Y, stream=None) -> None:
    """Y[M,N] (bf16) = dq(Xq, Xs) dq(Wq, Ws)^T."""
    import torch
    for t, n in ((Xq, "Xq"), (Xs, "Xs"), (Wq, "Wq"), (Ws, "Ws")):
        _require(t, torch.uint8, n, 2)
    _require(Y, torch.bfloat16, "Y", 2)
    M, K = Xq.shape
    N = Wq.shape[0]
    if Wq.shape[1] != K or tuple(Xs.shape) != (M, K // 32) or tuple(Ws.shape) != (N, K // 32) \
            or tuple(Y.shape) != (M, N):
        raise ValueError("shape mismatch")
    _check(lib().gtp_linear_fprop_mxfp8(_ptr(Xq), _ptr(Xs), _ptr(Wq), _ptr(Ws), _ptr(Y), M, N, K, _stream(stream)),
           "gtp_linear_fprop_mxfp8")


def gtp_wait_timeouts(reset: bool = False) -> int:
    """The per-device word of timed-out waits in the tensor-core kernels (0 = none)."""
    v = C.c_uint32(0)
    _check(lib().gtp_wait_timeouts(C.byref(v), int(reset)), "gtp_wait_timeouts")
    return v.value


def gtp_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    """Launches the bounded-wait self-test: one thread waits limit_ns on an mbarrier that
    nothing arrives on, gives up, sets bit 8 of the wait-timeout word and returns."""
    _check(lib().gtp_selftest_wait_timeout(int(limit_ns), _stream(stream)), "gtp_selftest_wait_timeout")


def gtp_grad_norm_noalloc(grad_data, buckets, factors: Sequence[float], max_norm: float, sumsq, nonfinite,
                          total_norm, clip_coef, stream=None) -> None:
    """gtp_grad_norm with the library's fixed scratch instead of a workspace (see include/gtp.h)."""
    import torch
    _require(grad_data, torch.float32, "grad_data")
    _require(sumsq, torch.float64, "sumsq")
    _require(nonfinite, torch.int32, "nonfinite")
    _require(total_norm, torch.float32, "total_norm")
    _require(clip_coef, torch.float32, "clip_coef")
    arr, nb = _bucket_args(buckets, factors)
    if sumsq.numel() < nb or nonfinite.numel() < nb:
        raise ValueError("sumsq and nonfinite need one entry per bucket")
    _check(lib().gtp_grad_norm_noalloc(_ptr(grad_data), grad_data.numel(), arr, _factor_array(factors), nb,
                                       float(max_norm), _ptr(sumsq), _ptr(nonfinite), _ptr(total_norm),
                                       _ptr(clip_coef), _stream(stream)),
           "gtp_grad_norm_noalloc")


def _col_args(src, e4m3_t, e8m0_t, tiled: bool = False):
    import torch
    dt = {torch.float32: abi.GTP_F32, torch.bfloat16: abi.GTP_BF16}.get(src.dtype)
    if dt is None:
        raise TypeError("src must be float32 or bfloat16")
    _require(src, src.dtype, "src", 2)
    R, Cc = src.shape
    _require(e4m3_t, torch.uint8, "e4m3_t", 2)
    if tuple(e4m3_t.shape) != (Cc, R):
        raise ValueError("e4m3_t must be [C,R]")
    if tiled:
        _require_tiled(e8m0_t, Cc, R // 32, "e8m0_t_tiled")
    else:
        _require(e8m0_t, torch.uint8, "e8m0_t", 2)
        if tuple(e8m0_t.shape) != (Cc, R // 32):
            raise ValueError("e8m0_t must be [C,R/32]")
    return dt, R, Cc


def gtp_mxfp8_quantize_columnwise(src, e4m3_t, e8m0_t, stream=None) -> None:
    """src[R,C] (fp32 or bf16) -> e4m3_t[C,R], e8m0_t[C,R/32]: blocks of 32 rows per column, transposed."""
    dt, R, Cc = _col_args(src, e4m3_t, e8m0_t)
    _check(lib().gtp_mxfp8_quantize_columnwise(_ptr(src), dt, R, Cc, _ptr(e4m3_t), _ptr(e8m0_t), _stream(stream)),
           "gtp_mxfp8_quantize_columnwise")


def gtp_mxfp8_quantize_columnwise_tiled(src, e4m3_t, e8m0_t_tiled, stream=None) -> None:
    """src[R,C] (fp32 or bf16) -> e4m3_t[C,R] and the [C,R/32] scales in the tiled layout."""
    dt, R, Cc = _col_args(src, e4m3_t, e8m0_t_tiled, tiled=True)
    _check(lib().gtp_mxfp8_quantize_columnwise_tiled(_ptr(src), dt, R, Cc, _ptr(e4m3_t), _ptr(e8m0_t_tiled),
                                                     _stream(stream)),
           "gtp_mxfp8_quantize_columnwise_tiled")


def gtp_mxfp8_quantize_columnwise_group(views: Sequence, stream=None) -> None:
    """Up to eight (src, e4m3_t, e8m0_t) triples, each as gtp_mxfp8_quantize_columnwise (a
    2-D e8m0_t [C,R/32]) or gtp_mxfp8_quantize_columnwise_tiled (a 1-D tiled e8m0_t), in
    one launch."""
    descs = []
    for src, q, s in views:
        tiled = s.dim() == 1
        dt, R, Cc = _col_args(src, q, s, tiled)
        descs.append(abi.gtp_mx_col_desc(_ptr(src), _ptr(q), _ptr(s), R, Cc, dt, int(tiled)))
    arr = (abi.gtp_mx_col_desc * max(len(descs), 1))(*descs)
    _check(lib().gtp_mxfp8_quantize_columnwise_group(arr, len(descs), _stream(stream)),
           "gtp_mxfp8_quantize_columnwise_group")


def gtp_linear_dgrad_mxfp8(dYq, dYs, Wtq, Wts, dX, stream=None) -> None:
    """dX[M,K] (bf16) = dq(dYq[M,N], dYs) dq(Wtq[K,N], Wts)^T."""
    import torch
    for t, n in ((dYq, "dYq"), (dYs, "dYs"), (Wtq, "Wtq"), (Wts, "Wts")):
        _require(t, torch.uint8, n, 2)
    _require(dX, torch.bfloat16, "dX", 2)
    M, N = dYq.shape
    K = Wtq.shape[0]
    if Wtq.shape[1] != N or tuple(dYs.shape) != (M, N // 32) or tuple(Wts.shape) != (K, N // 32) \
            or tuple(dX.shape) != (M, K):
        raise ValueError("shape mismatch")
    _check(lib().gtp_linear_dgrad_mxfp8(_ptr(dYq), _ptr(dYs), _ptr(Wtq), _ptr(Wts), _ptr(dX), M, N, K,
                                        _stream(stream)),
           "gtp_linear_dgrad_mxfp8")


def gtp_linear_wgrad_accum_mxfp8(dYtq, dYts, Xtq, Xts, grad_data, grad_offset: int, stream=None) -> None:
    """grad_data[grad_offset:+N*K].view(N,K) += dq(dYtq[N,M], dYts) dq(Xtq[K,M], Xts)^T (fp32)."""
    import torch
    for t, n in ((dYtq, "dYtq"), (dYts, "dYts"), (Xtq, "Xtq"), (Xts, "Xts")):
        _require(t, torch.uint8, n, 2)
    _require(grad_data, torch.float32, "grad_data")
    N, M = dYtq.shape
    K = Xtq.shape[0]
    if Xtq.shape[1] != M or tuple(dYts.shape) != (N, M // 32) or tuple(Xts.shape) != (K, M // 32):
        raise ValueError("shape mismatch")
    _check(lib().gtp_linear_wgrad_accum_mxfp8(_ptr(dYtq), _ptr(dYts), _ptr(Xtq), _ptr(Xts), _ptr(grad_data),
                                              int(grad_offset), grad_data.numel(), M, N, K, _stream(stream)),
           "gtp_linear_wgrad_accum_mxfp8")


def gtp_rs_local_sum(slices, out, stream=None) -> None:
    """out = the fp32 sum, in rank order, of the received slices, cast to out's dtype: the
    local half of the all-to-all reduce-scatter with fp32 accumulation.  slices: the
    all-to-all's receive buffer as one contiguous [P, n] tensor (row r from rank r), or a
    sequence of P 1-D tensors of n elements; bf16 or fp32."""
    import torch
    dts = {torch.float32: abi.GTP_F32, torch.bfloat16: abi.GTP_BF16}
    if out.dtype not in dts:
        raise TypeError("out must be float32 or bfloat16")
    _require(out, out.dtype, "out", 1)
    n = out.numel()
    if isinstance(slices, torch.Tensor):
        if slices.dtype not in dts:
            raise TypeError("slices must be float32 or bfloat16")
        _require(slices, slices.dtype, "slices", 2)
        if slices.shape[1] != n or slices.shape[0] < 1:
            raise ValueError("slices must be [P, n] with n = out's length")
        _check(lib().gtp_rs_local_sum_rows(_ptr(slices), n * slices.element_size(), slices.shape[0], n,
                                           dts[slices.dtype], _ptr(out), dts[out.dtype], _stream(stream)),
               "gtp_rs_local_sum_rows")
        return
    if not slices:
        raise ValueError("at least one slice")
    in_dt, P = slices[0].dtype, len(slices)
    if in_dt not in dts:
        raise TypeError("slices must be float32 or bfloat16")
    for i, t in enumerate(slices):
        _require(t, in_dt, f"slices[{i}]", 1)
        if t.numel() != n:
            raise ValueError("every slice has out's length")
    arr = (C.c_void_p * P)(*[_ptr(t) for t in slices])
    _check(lib().gtp_rs_local_sum(arr, P, n, dts[in_dt], _ptr(out), dts[out.dtype], _stream(stream)),
           "gtp_rs_local_sum")


# ----------------------------------------------------------------------------- NVFP4

def gtp_nvfp4_quantize_rowwise(src, packed, scales, amax, stream=None) -> None:
    """src[R,C] (fp32 or bf16) -> packed[R,C/2], scales[R,C/16] (uint8) and amax[1] (fp32)."""
    import torch
    dt = {torch.float32: abi.GTP_F32, torch.bfloat16: abi.GTP_BF16}.get(src.dtype)
    if dt is None:
        raise TypeError("src must be float32 or bfloat16")
    _require(src, src.dtype, "src", 2)
    R, Cc = src.shape
    _require(packed, torch.uint8, "packed", 2)
    _require(scales, torch.uint8, "scales", 2)
    _require(amax, torch.float32, "amax")
    if tuple(packed.shape) != (R, Cc // 2) or tuple(scales.shape) != (R, Cc // 16) or amax.numel() != 1:
        raise ValueError("packed must be [R,C/2], scales [R,C/16] and amax one element")
    _check(lib().gtp_nvfp4_quantize_rowwise(_ptr(src), dt, R, Cc, _ptr(packed), _ptr(scales), _ptr(amax),
                                            _stream(stream)),
           "gtp_nvfp4_quantize_rowwise")


def gtp_linear_fprop_nvfp4(Xq, Xs, x_amax, Wq, Ws, w_amax, Y, stream=None) -> None:
    """Y[M,N] (bf16) = dq(Xq, Xs, x_amax) dq(Wq, Ws, w_amax)^T, operands packed [rows, K/2]."""
    import torch
    for t, n in ((Xq, "Xq"), (Xs, "Xs"), (Wq, "Wq"), (Ws, "Ws")):
        _require(t, torch.uint8, n, 2)
    for t, n in ((x_amax, "x_amax"), (w_amax, "w_amax")):
        _require(t, torch.float32, n)
    _require(Y, torch.bfloat16, "Y", 2)
    M, K = Xq.shape[0], Xq.shape[1] * 2
    N = Wq.shape[0]
    if Wq.shape[1] * 2 != K or tuple(Xs.shape) != (M, K // 16) or tuple(Ws.shape) != (N, K // 16) \
            or tuple(Y.shape) != (M, N):
        raise ValueError("shape mismatch")
    _check(lib().gtp_linear_fprop_nvfp4(_ptr(Xq), _ptr(Xs), _ptr(x_amax), _ptr(Wq), _ptr(Ws), _ptr(w_amax), _ptr(Y),
                                        M, N, K, _stream(stream)),
           "gtp_linear_fprop_nvfp4")


# ----------------------------------------------------------------------------- tiled scale layout

def gtp_sf_tiled_bytes(rows: int, cols: int) -> int:
    """Bytes of the tiled form of a [rows, cols] scale array (host only)."""
    n = lib().gtp_sf_tiled_bytes(int(rows), int(cols))
    if n < 0:
        raise ValueError("negative size")
    return n


def _require_tiled(t, rows: int, cols: int, name: str) -> None:
    import torch
    _require(t, torch.uint8, name)
    if t.numel() != gtp_sf_tiled_bytes(rows, cols):
        raise ValueError(f"{name} must hold gtp_sf_tiled_bytes({rows}, {cols}) bytes")


def gtp_sf_tile(sf, tiled, stream=None) -> None:
    """sf[R,C] (uint8 scale bytes) -> tiled (uint8, gtp_sf_tiled_bytes(R, C) bytes)."""
    import torch
    _require(sf, torch.uint8, "sf", 2)
    R, Cc = sf.shape
    _require_tiled(tiled, R, Cc, "tiled")
    _check(lib().gtp_sf_tile(_ptr(sf), R, Cc, _ptr(tiled), _stream(stream)), "gtp_sf_tile")


def gtp_mxfp8_quantize_rowwise_tiled(src, e4m3, e8m0_tiled, stream=None) -> None:
    """src[R,C] (fp32 or bf16) -> e4m3[R,C] and the [R,C/32] scales in the tiled layout."""
    import torch
    dt = {torch.float32: abi.GTP_F32, torch.bfloat16: abi.GTP_BF16}.get(src.dtype)
    if dt is None:
        raise TypeError("src must be float32 or bfloat16")
    _require(src, src.dtype, "src", 2)
    R, Cc = src.shape
    _require(e4m3, torch.uint8, "e4m3", 2)
    if tuple(e4m3.shape) != (R, Cc):
        raise ValueError("e4m3 must be [R,C]")
    _require_tiled(e8m0_tiled, R, Cc // 32, "e8m0_tiled")
    _check(lib().gtp_mxfp8_quantize_rowwise_tiled(_ptr(src), dt, R, Cc, _ptr(e4m3), _ptr(e8m0_tiled),
                                                  _stream(stream)),
           "gtp_mxfp8_quantize_rowwise_tiled")


def gtp_nvfp4_quantize_rowwise_tiled(src, packed, scales_tiled, amax, stream=None) -> None:
    """src[R,C] (fp32 or bf16) -> packed[R,C/2], the [R,C/16] scales in the tiled layout, amax[1]."""
    import torch
    dt = {torch.float32: abi.GTP_F32, torch.bfloat16: abi.GTP_BF16}.get(src.dtype)
    if dt is None:
        raise TypeError("src must be float32 or bfloat16")
    _require(src, src.dtype, "src", 2)
    R, Cc = src.shape
    _require(packed, torch.uint8, "packed", 2)
    _require(amax, torch.float32, "amax")
    if tuple(packed.shape) != (R, Cc // 2) or amax.numel() != 1:
        raise ValueError("packed must be [R,C/2] and amax one element")
    _require_tiled(scales_tiled, R, Cc // 16, "scales_tiled")
    _check(lib().gtp_nvfp4_quantize_rowwise_tiled(_ptr(src), dt, R, Cc, _ptr(packed), _ptr(scales_tiled),
                                                  _ptr(amax), _stream(stream)),
           "gtp_nvfp4_quantize_rowwise_tiled")


def gtp_linear_fprop_mxfp8_tiled(Xq, Xs_tiled, Wq, Ws_tiled, Y, stream=None) -> None:
    """Y[M,N] (bf16) = dq(Xq, Xs) dq(Wq, Ws)^T with both scale arrays in the tiled layout."""
    import torch
    for t, n in ((Xq, "Xq"), (Wq, "Wq")):
        _require(t, torch.uint8, n, 2)
    _require(Y, torch.bfloat16, "Y", 2)
    M, K = Xq.shape
    N = Wq.shape[0]
    if Wq.shape[1] != K or tuple(Y.shape) != (M, N):
        raise ValueError("shape mismatch")
    _require_tiled(Xs_tiled, M, K // 32, "Xs_tiled")
    _require_tiled(Ws_tiled, N, K // 32, "Ws_tiled")
    _check(lib().gtp_linear_fprop_mxfp8_tiled(_ptr(Xq), _ptr(Xs_tiled), _ptr(Wq), _ptr(Ws_tiled), _ptr(Y), M, N, K,
                                              _stream(stream)),
           "gtp_linear_fprop_mxfp8_tiled")


def gtp_linear_dgrad_mxfp8_tiled(dYq, dYs_tiled, Wtq, Wts_tiled, dX, stream=None) -> None:
    """dX[M,K] (bf16) = dq(dYq[M,N], dYs) dq(Wtq[K,N], Wts)^T, both scale arrays in the tiled layout."""
    import torch
    for t, n in ((dYq, "dYq"), (Wtq, "Wtq")):
        _require(t, torch.uint8, n, 2)
    _require(dX, torch.bfloat16, "dX", 2)
    M, N = dYq.shape
    K = Wtq.shape[0]
    if Wtq.shape[1] != N or tuple(dX.shape) != (M, K):
        raise ValueError("shape mismatch")
    _require_tiled(dYs_tiled, M, N // 32, "dYs_tiled")
    _require_tiled(Wts_tiled, K, N // 32, "Wts_tiled")
    _check(lib().gtp_linear_dgrad_mxfp8_tiled(_ptr(dYq), _ptr(dYs_tiled), _ptr(Wtq), _ptr(Wts_tiled), _ptr(dX), M, N,
                                              K, _stream(stream)),
           "gtp_linear_dgrad_mxfp8_tiled")


def gtp_linear_wgrad_accum_mxfp8_tiled(dYtq, dYts_tiled, Xtq, Xts_tiled, grad_data, grad_offset: int,
                                       stream=None) -> None:
    """grad_data[grad_offset:+N*K].view(N,K) += dq(dYtq[N,M], dYts) dq(Xtq[K,M], Xts)^T (fp32), both
    scale arrays in the tiled layout."""
    import torch
    for t, n in ((dYtq, "dYtq"), (Xtq, "Xtq")):
        _require(t, torch.uint8, n, 2)
    _require(grad_data, torch.float32, "grad_data")
    N, M = dYtq.shape
    K = Xtq.shape[0]
    if Xtq.shape[1] != M:
        raise ValueError("shape mismatch")
    _require_tiled(dYts_tiled, N, M // 32, "dYts_tiled")
    _require_tiled(Xts_tiled, K, M // 32, "Xts_tiled")
    _check(lib().gtp_linear_wgrad_accum_mxfp8_tiled(_ptr(dYtq), _ptr(dYts_tiled), _ptr(Xtq), _ptr(Xts_tiled),
                                                    _ptr(grad_data), int(grad_offset), grad_data.numel(), M, N, K,
                                                    _stream(stream)),
           "gtp_linear_wgrad_accum_mxfp8_tiled")


def gtp_linear_fprop_nvfp4_tiled(Xq, Xs_tiled, x_amax, Wq, Ws_tiled, w_amax, Y, stream=None) -> None:
    """Y[M,N] (bf16) = dq(Xq, Xs, x_amax) dq(Wq, Ws, w_amax)^T, scale arrays in the tiled layout."""
    import torch
    for t, n in ((Xq, "Xq"), (Wq, "Wq")):
        _require(t, torch.uint8, n, 2)
    for t, n in ((x_amax, "x_amax"), (w_amax, "w_amax")):
        _require(t, torch.float32, n)
    _require(Y, torch.bfloat16, "Y", 2)
    M, K = Xq.shape[0], Xq.shape[1] * 2
    N = Wq.shape[0]
    if Wq.shape[1] * 2 != K or tuple(Y.shape) != (M, N):
        raise ValueError("shape mismatch")
    _require_tiled(Xs_tiled, M, K // 16, "Xs_tiled")
    _require_tiled(Ws_tiled, N, K // 16, "Ws_tiled")
    _check(lib().gtp_linear_fprop_nvfp4_tiled(_ptr(Xq), _ptr(Xs_tiled), _ptr(x_amax), _ptr(Wq), _ptr(Ws_tiled),
                                              _ptr(w_amax), _ptr(Y), M, N, K, _stream(stream)),
           "gtp_linear_fprop_nvfp4_tiled")
