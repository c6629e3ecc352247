"""ctypes view of ``include/gtp.h``: structs, enums and function prototypes of libgtp.so.

This module only loads the shared library and declares its C signatures.  It never
computes anything; a missing library is an error (``LibraryNotBuilt``), never a
fallback.
"""
from __future__ import annotations

import ctypes as C
from pathlib import Path

LIB_PATH = Path(__file__).resolve().parent / "libgtp.so"

# gtp_status
GTP_OK, GTP_E_ARG, GTP_E_SHAPE, GTP_E_ALIGN, GTP_E_DTYPE, GTP_E_RANGE, GTP_E_CAPACITY, GTP_E_CUDA, GTP_E_DEVICE = range(9)
STATUS_NAMES = {
    0: "GTP_OK", 1: "GTP_E_ARG", 2: "GTP_E_SHAPE", 3: "GTP_E_ALIGN", 4: "GTP_E_DTYPE",
    5: "GTP_E_RANGE", 6: "GTP_E_CAPACITY", 7: "GTP_E_CUDA", 8: "GTP_E_DEVICE",
}
# gtp_dtype
GTP_F32, GTP_BF16, GTP_F16, GTP_U8 = 0, 1, 2, 3


class gtp_param_desc(C.Structure):
    _fields_ = [("numel", C.c_int64), ("dtype", C.c_int32), ("quantized_storage", C.c_int32),
                ("is_expert_parallel", C.c_int32), ("is_layer_wise", C.c_int32),
                ("is_shared_embedding", C.c_int32), ("reserved", C.c_int32)]


class gtp_layout_config(C.Structure):
    _fields_ = [("bucket_size", C.c_int64), ("dp_size", C.c_int32),
                ("use_distributed_optimizer", C.c_int32),
                ("pad_buckets_for_high_nccl_busbw", C.c_int32), ("grad_reduce_in_fp32", C.c_int32)]


class gtp_param_index(C.Structure):
    _fields_ = [("start", C.c_int64), ("end", C.c_int64), ("start_in_bucket", C.c_int64),
                ("end_in_bucket", C.c_int64), ("bucket_id", C.c_int32), ("buffer_id", C.c_int32)]


class gtp_bucket_desc(C.Structure):
    _fields_ = [("offset", C.c_int64), ("numel_unpadded", C.c_int64), ("numel", C.c_int64),
                ("buffer_id", C.c_int32), ("num_params", C.c_int32)]


class gtp_buffer_desc(C.Structure):
    _fields_ = [("numel", C.c_int64), ("param_dtype", C.c_int32), ("grad_dtype", C.c_int32),
                ("is_expert_parallel", C.c_int32), ("is_layer_wise", C.c_int32),
                ("first_bucket", C.c_int32), ("num_buckets", C.c_int32)]


class gtp_shard_range(C.Structure):
    _fields_ = [("param", C.c_int32), ("bucket_id", C.c_int32), ("world_start", C.c_int64),
                ("world_end", C.c_int64), ("bucket_start", C.c_int64), ("local_start", C.c_int64),
                ("param_start", C.c_int64)]


class gtp_mx_col_desc(C.Structure):
    _fields_ = [("src", C.c_void_p), ("e4m3_t", C.c_void_p), ("e8m0_t", C.c_void_p), ("rows", C.c_int64),
                ("cols", C.c_int64), ("src_dtype", C.c_int32), ("tiled_scales", C.c_int32)]


class gtp_mx_row_desc(C.Structure):
    _fields_ = [("src", C.c_void_p), ("e4m3", C.c_void_p), ("e8m0", C.c_void_p), ("rows", C.c_int64),
                ("cols", C.c_int64), ("src_dtype", C.c_int32), ("tiled_scales", C.c_int32)]


class gtp_gemm_desc(C.Structure):
    _fields_ = [("kind", C.c_int32), ("dtype", C.c_int32), ("a", C.c_void_p), ("b", C.c_void_p),
                ("out", C.c_void_p), ("M", C.c_int64), ("N", C.c_int64), ("K", C.c_int64),
                ("grad_offset", C.c_int64), ("grad_numel_total", C.c_int64),
                ("grad_dtype", C.c_int32), ("reserved", C.c_int32)]


GTP_GEMM_FPROP, GTP_GEMM_DGRAD, GTP_GEMM_WGRAD_ACCUM = 0, 1, 2
GTP_GEMM_DETERMINISTIC = 1


class gtp_adam_hparams(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float),
                ("weight_decay", C.c_float), ("zero_grad_after", C.c_int32), ("step", C.c_int64),
                ("grad_scale", C.c_void_p)]


VP, I64, I32 = C.c_void_p, C.c_int64, C.c_int32
P = C.POINTER

# name -> (restype, argtypes); every entry point declared in include/gtp.h
PROTOTYPES = {
    "gtp_last_error": (C.c_char_p, []),
    "gtp_linear_fprop": (I32, [VP, VP, VP, I64, I64, I64, I32, VP]),
    "gtp_linear_dgrad": (I32, [VP, VP, VP, I64, I64, I64, I32, VP]),
    "gtp_linear_wgrad_accum": (I32, [VP, VP, VP, I64, I64, I64, I64, I64, I32, VP]),
    "gtp_linear_wgrad_accum_deterministic": (I32, [VP, VP, VP, I64, I64, I64, I64, I64, I32, VP]),
    "gtp_linear_wgrad_accum_bf16": (I32, [VP, VP, VP, I64, I64, I64, I64, I64, I32, VP]),
    "gtp_linear_grouped": (I32, [P(gtp_gemm_desc), I32, I32, VP]),
    "gtp_linear_backward": (I32, [VP, VP, VP, VP, VP, I64, I64, I64, I64, I64, I32, I32, VP]),
    "gtp_buffer_layout": (I32, [P(gtp_param_desc), I32, P(gtp_layout_config), P(gtp_param_index),
                                P(gtp_buffer_desc), P(I32), P(gtp_bucket_desc), P(I32)]),
    "gtp_shard_param_ranges": (I32, [P(gtp_param_index), I32, P(gtp_bucket_desc), I32, I32, I32, I32,
                                     P(gtp_shard_range), P(I32)]),
    "gtp_buffer_zero": (I32, [VP, I32, I64, VP]),
    "gtp_bucket_scale": (I32, [VP, I64, P(gtp_bucket_desc), P(C.c_float), I32, VP]),
    "gtp_adam_step_flat": (I32, [VP, VP, VP, VP, VP, I64, P(gtp_bucket_desc), P(C.c_float), I32,
                                 P(gtp_adam_hparams), VP]),
    "gtp_adam_step_flat_mxfp8": (I32, [VP, VP, VP, VP, VP, VP, I64, P(gtp_bucket_desc), P(C.c_float), I32,
                                       P(gtp_adam_hparams), VP]),
    "gtp_adam_step_flat_bf16_grad": (I32, [VP, VP, VP, VP, VP, I64, P(gtp_bucket_desc), P(C.c_float), I32,
                                           P(gtp_adam_hparams), VP]),
    "gtp_mxfp8_quantize_rowwise": (I32, [VP, I32, I64, I64, VP, VP, VP]),
    "gtp_linear_fprop_mxfp8": (I32, [VP, VP, VP, VP, VP, I64, I64, I64, VP]),
    "gtp_mxfp8_quantize_columnwise": (I32, [VP, I32, I64, I64, VP, VP, VP]),
    "gtp_mxfp8_quantize_columnwise_group": (I32, [P(gtp_mx_col_desc), I32, VP]),
    "gtp_mxfp8_quantize_columnwise_tiled": (I32, [VP, I32, I64, I64, VP, VP, VP]),
    "gtp_mxfp8_quantize_rowwise_group": (I32, [P(gtp_mx_row_desc), I32, VP]),
    "gtp_rs_local_sum": (I32, [P(VP), I32, I64, I32, VP, I32, VP]),
    "gtp_rs_local_sum_rows": (I32, [VP, I64, I32, I64, I32, VP, I32, VP]),
    "gtp_linear_dgrad_mxfp8": (I32, [VP, VP, VP, VP, VP, I64, I64, I64, VP]),
    "gtp_linear_wgrad_accum_mxfp8": (I32, [VP, VP, VP, VP, VP, I64, I64, I64, I64, I64, VP]),
    "gtp_nvfp4_quantize_rowwise": (I32, [VP, I32, I64, I64, VP, VP, VP, VP]),
    "gtp_linear_fprop_nvfp4": (I32, [VP, VP, VP, VP, VP, VP, VP, I64, I64, I64, VP]),
    "gtp_sf_tiled_bytes": (I64, [I64, I64]),
    "gtp_sf_tile": (I32, [VP, I64, I64, VP, VP]),
    "gtp_mxfp8_quantize_rowwise_tiled": (I32, [VP, I32, I64, I64, VP, VP, VP]),
    "gtp_nvfp4_quantize_rowwise_tiled": (I32, [VP, I32, I64, I64, VP, VP, VP, VP]),
    "gtp_linear_fprop_mxfp8_tiled": (I32, [VP, VP, VP, VP, VP, I64, I64, I64, VP]),
    "gtp_linear_dgrad_mxfp8_tiled": (I32, [VP, VP, VP, VP, VP, I64, I64, I64, VP]),
    "gtp_linear_wgrad_accum_mxfp8_tiled": (I32, [VP, VP, VP, VP, VP, I64, I64, I64, I64, I64, VP]),
    "gtp_linear_fprop_nvfp4_tiled": (I32, [VP, VP, VP, VP, VP, VP, VP, I64, I64, I64, VP]),
    "gtp_wait_timeouts": (I32, [P(C.c_uint32), I32]),
    "gtp_selftest_wait_timeout": (I32, [I64, VP]),
    "gtp_grad_norm_workspace_bytes": (C.c_size_t, [P(gtp_bucket_desc), I32]),
    "gtp_grad_norm": (I32, [VP, I64, P(gtp_bucket_desc), P(C.c_float), I32, C.c_float, VP, C.c_size_t, VP, VP,
                            VP, VP, VP]),
    "gtp_grad_norm_noalloc": (I32, [VP, I64, P(gtp_bucket_desc), P(C.c_float), I32, C.c_float, VP, VP, VP, VP,
                                    VP]),
}


class LibraryNotBuilt(RuntimeError):
    pass


_lib = None


def load(path: Path | str | None = None) -> C.CDLL:
    """Loads libgtp.so (once) and declares every prototype; raises if it is absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path else LIB_PATH
    if not p.exists():
        raise LibraryNotBuilt(f"{p} is missing: run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = C.CDLL(str(p))
    for name, (res, args) in PROTOTYPES.items():
        try:
            fn = getattr(lib, name)
        except AttributeError:
            continue  # calling it raises AttributeError; tests/test_abi.py requires every symbol
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib
