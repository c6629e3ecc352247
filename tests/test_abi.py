"""The C ABI without a GPU: the library loads, exports every declared entry point, and
rejects bad arguments on the host before touching a device.

Every call below is built so that host-side validation must reject it; none of them
reaches a CUDA call, so the fake addresses used for alignment checks are never
dereferenced.
"""
import ctypes as C
import re
from pathlib import Path

import pytest

from param_buffers_gb300 import abi

ROOT = Path(__file__).resolve().parents[1]
pytestmark = pytest.mark.skipif(not abi.LIB_PATH.exists(), reason="libgtp.so not built")


def declared_functions():
    text = (ROOT / "include" / "gtp.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gtp_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported_and_bound():
    lib = abi.load()
    names = declared_functions()
    assert "gtp_linear_wgrad_accum" in names and "gtp_adam_step_flat" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(abi.PROTOTYPES), set(names) - set(abi.PROTOTYPES)


def test_struct_sizes_match_header_layout():
    assert C.sizeof(abi.gtp_param_desc) == 32
    assert C.sizeof(abi.gtp_layout_config) == 24
    assert C.sizeof(abi.gtp_param_index) == 40
    assert C.sizeof(abi.gtp_bucket_desc) == 32
    assert C.sizeof(abi.gtp_buffer_desc) == 32
    assert C.sizeof(abi.gtp_adam_hparams) == 40


MISALIGNED = 0x1004       # never dereferenced: every call using it fails validation first
ALIGNED = 0x100000


def test_sweep_argument_errors():
    lib = abi.load()
    h = abi.gtp_adam_hparams(3e-4, 0.9, 0.95, 1e-8, 0.1, 1, 1)
    assert lib.gtp_buffer_zero(None, abi.GTP_F32, 10, None) == abi.GTP_E_ARG
    assert lib.gtp_buffer_zero(MISALIGNED, abi.GTP_F32, 10, None) == abi.GTP_E_ALIGN
    assert lib.gtp_buffer_zero(ALIGNED, 9, 10, None) == abi.GTP_E_DTYPE
    assert lib.gtp_buffer_zero(ALIGNED, abi.GTP_F32, -1, None) == abi.GTP_E_ARG
    assert lib.gtp_buffer_zero(None, abi.GTP_F32, 0, None) == abi.GTP_OK      # empty: nothing to do
    bk = (abi.gtp_bucket_desc * 2)(abi.gtp_bucket_desc(0, 100, 100, 0, 1), abi.gtp_bucket_desc(50, 100, 100, 0, 1))
    fac = (C.c_float * 2)(0.5, 0.5)
    assert lib.gtp_bucket_scale(ALIGNED, 1000, bk, fac, 2, None) == abi.GTP_E_RANGE          # overlap
    assert b"overlaps" in lib.gtp_last_error()
    bk2 = (abi.gtp_bucket_desc * 1)(abi.gtp_bucket_desc(990, 100, 100, 0, 1))
    assert lib.gtp_bucket_scale(ALIGNED, 1000, bk2, fac, 1, None) == abi.GTP_E_RANGE         # past the end
    assert lib.gtp_bucket_scale(MISALIGNED, 1000, bk2, fac, 1, None) == abi.GTP_E_ALIGN
    assert lib.gtp_bucket_scale(ALIGNED, 1000, None, fac, 1, None) == abi.GTP_E_ARG
    many = (abi.gtp_bucket_desc * 513)()
    manyf = (C.c_float * 513)()
    assert lib.gtp_bucket_scale(ALIGNED, 10 ** 6, many, manyf, 513, None) == abi.GTP_E_CAPACITY
    ptrs = [ALIGNED + k * (1 << 24) for k in range(5)]   # distinct arrays (the sweep refuses overlaps)
    assert lib.gtp_adam_step_flat(*ptrs, 100, None, None, 0, None, None) == abi.GTP_E_ARG
    assert lib.gtp_adam_step_flat(*ptrs[:4], MISALIGNED, 100, None, None, 0, C.byref(h), None) == abi.GTP_E_ALIGN
    assert lib.gtp_adam_step_flat(None, *ptrs[1:], 100, None, None, 0, C.byref(h), None) == abi.GTP_E_ARG
    for bad in (abi.gtp_adam_hparams(3e-4, 1.0, 0.95, 1e-8, 0.1, 1, 1),
                abi.gtp_adam_hparams(3e-4, 0.9, 0.95, 1e-8, 0.1, 1, 0),
                abi.gtp_adam_hparams(-1.0, 0.9, 0.95, 1e-8, 0.1, 1, 1),
                abi.gtp_adam_hparams(3e-4, 0.9, 0.95, float("nan"), 0.1, 1, 1),
                abi.gtp_adam_hparams(3e-4, 0.9, 0.95, 1e-8, 0.1, 2, 1)):
        assert lib.gtp_adam_step_flat(*ptrs, 100, None, None, 0, C.byref(bad), None) == abi.GTP_E_ARG
    assert lib.gtp_adam_step_flat(*ptrs, 1000, bk, fac, 2, C.byref(h), None) == abi.GTP_E_RANGE
    # the native-MXFP8 sweep: whole 32-element blocks, aligned codes, both outputs
    mx = [ALIGNED + k * (1 << 24) for k in range(6)]
    assert lib.gtp_adam_step_flat_mxfp8(*mx, 100, None, None, 0, C.byref(h), None) == abi.GTP_E_SHAPE
    assert lib.gtp_adam_step_flat_mxfp8(*mx[:4], MISALIGNED, ALIGNED, 128, None, None, 0, C.byref(h),
                                        None) == abi.GTP_E_ALIGN
    assert lib.gtp_adam_step_flat_mxfp8(*mx[:5], None, 128, None, None, 0, C.byref(h), None) == abi.GTP_E_ARG
    assert lib.gtp_adam_step_flat_mxfp8(*mx[:5], mx[5] + 2, 128, None, None, 0, C.byref(h), None) == abi.GTP_E_ALIGN
    assert lib.gtp_adam_step_flat_mxfp8(*mx, 1024, bk, fac, 2, C.byref(h), None) == abi.GTP_E_RANGE
    assert lib.gtp_adam_step_flat_mxfp8(*mx, 128, None, None, 0, None, None) == abi.GTP_E_ARG
    assert lib.gtp_adam_step_flat_mxfp8(None, None, None, None, None, None, 0, None, None, 0, C.byref(h),
                                        None) == abi.GTP_OK


def test_noalloc_grad_norm_rejects_inputs_beyond_its_scratch():
    """The non-allocating gradient norm refuses, on the host and before any CUDA call, an
    input with more chunk partials than its fixed scratch array holds."""
    lib = abi.load()
    too_many = 65536 * 65536 + 1                        # one chunk more than the scratch holds
    b = (abi.gtp_bucket_desc * 1)(abi.gtp_bucket_desc(0, too_many, too_many, 0, 1))
    st = lib.gtp_grad_norm_noalloc(ALIGNED, too_many, b, (C.c_float * 1)(1.0), 1, 1.0,
                                   ALIGNED, ALIGNED, ALIGNED, ALIGNED, None)
    assert st == abi.GTP_E_CAPACITY
    assert b"fixed scratch" in lib.gtp_last_error()


def test_grad_norm_wrappers_check_outputs_and_factor_count():
    """The Python bindings reject a wrong output dtype, a short output and a factor list
    whose length differs from the bucket count before calling into the library."""
    import torch
    import param_buffers_gb300 as gtp
    g = torch.zeros(64)
    b = [{"offset": 0, "numel": 32}, {"offset": 32, "numel": 32}]
    good = [torch.zeros(2, dtype=torch.float64), torch.zeros(2, dtype=torch.int32),
            torch.zeros(1), torch.zeros(1)]
    bad_dtype = [torch.zeros(2, dtype=torch.float32)] + good[1:]
    short = [torch.zeros(1, dtype=torch.float64)] + good[1:]
    with pytest.raises(TypeError):
        gtp.gtp_grad_norm_noalloc(g, b, [1.0, 1.0], 1.0, *bad_dtype)
    with pytest.raises(ValueError):
        gtp.gtp_grad_norm_noalloc(g, b, [1.0, 1.0], 1.0, *short)
    with pytest.raises(ValueError):
        gtp.gtp_grad_norm_noalloc(g, b, [1.0], 1.0, *good)
    with pytest.raises(ValueError):
        gtp.gtp_grad_norm(g, b, [1.0], 1.0, torch.zeros(16, dtype=torch.uint8), *good)
    with pytest.raises(TypeError):
        gtp.gtp_grad_norm(g, b, [1.0, 1.0], 1.0, torch.zeros(16, dtype=torch.uint8), *bad_dtype)
    with pytest.raises(ValueError):
        gtp.gtp_bucket_scale(g, b, [0.5])


def test_wait_selftest_limit_is_checked_on_the_host():
    lib = abi.load()
    assert lib.gtp_selftest_wait_timeout(10, None) == abi.GTP_E_ARG            # below 1 us
    assert lib.gtp_selftest_wait_timeout(10 ** 9, None) == abi.GTP_E_ARG       # above 100 ms


def test_grouped_argument_errors_on_the_host():
    lib = abi.load()
    assert C.sizeof(abi.gtp_gemm_desc) == 80
    d = (abi.gtp_gemm_desc * 5)()
    assert lib.gtp_linear_grouped(d, 5, 0, None) == abi.GTP_E_ARG                 # more than four products
    assert lib.gtp_linear_grouped(None, 1, 0, None) == abi.GTP_E_ARG
    assert lib.gtp_linear_grouped(d, 1, 4, None) == abi.GTP_E_ARG                 # unknown flag
    d[0] = abi.gtp_gemm_desc(7, abi.GTP_BF16, ALIGNED, ALIGNED, ALIGNED, 256, 64, 64, 0, 0)
    assert lib.gtp_linear_grouped(d, 1, 0, None) == abi.GTP_E_ARG                 # unknown kind
    d[0] = abi.gtp_gemm_desc(abi.GTP_GEMM_FPROP, abi.GTP_F32, ALIGNED, ALIGNED, ALIGNED, 256, 64, 64, 0, 0)
    assert lib.gtp_linear_grouped(d, 1, 0, None) == abi.GTP_E_DTYPE
    d[0] = abi.gtp_gemm_desc(abi.GTP_GEMM_WGRAD_ACCUM, abi.GTP_BF16, ALIGNED, ALIGNED, 0x1002, 256, 64, 64, 2, 10 ** 6)
    assert lib.gtp_linear_grouped(d, 1, 0, None) == abi.GTP_E_ALIGN               # fp32 buffer not 4-byte aligned
    d[0].grad_dtype = abi.GTP_BF16
    d[0].out = 0x1001
    assert lib.gtp_linear_grouped(d, 1, 0, None) == abi.GTP_E_ALIGN               # bf16 buffer not 2-byte aligned
    d[0].grad_dtype = abi.GTP_F16
    assert lib.gtp_linear_grouped(d, 1, 0, None) == abi.GTP_E_DTYPE               # fp32 or bf16 grad buffers only
    d[0].grad_dtype = abi.GTP_BF16
    d[0].reserved = 1
    assert lib.gtp_linear_grouped(d, 1, 0, None) == abi.GTP_E_ARG                 # reserved must be 0
    assert lib.gtp_linear_grouped(d, 0, 0, None) == abi.GTP_OK                    # nothing to do
    assert lib.gtp_linear_backward(ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, 0, 100, 256, 64, 64, abi.GTP_BF16,
                                   0, None) == abi.GTP_E_RANGE                   # view larger than the buffer
    assert lib.gtp_linear_backward(ALIGNED, ALIGNED, ALIGNED, MISALIGNED, ALIGNED, 0, 10 ** 6, 256, 64, 64,
                                   abi.GTP_BF16, 0, None) == abi.GTP_E_ALIGN


def test_wgrad_view_alignment_rules_on_the_host():
    """Any element offset is accepted (a view TMA cannot address takes the register
    epilogue); the buffer itself must be aligned to its element."""
    lib = abi.load()
    args = (256, 64, 64, abi.GTP_BF16, None)
    assert lib.gtp_linear_wgrad_accum(ALIGNED, ALIGNED, 0x1002, 0, 10 ** 6, *args) == abi.GTP_E_ALIGN
    assert lib.gtp_linear_wgrad_accum_bf16(ALIGNED, ALIGNED, 0x1001, 0, 10 ** 6, *args) == abi.GTP_E_ALIGN
    assert lib.gtp_linear_wgrad_accum_bf16(ALIGNED, ALIGNED, ALIGNED, 5, 100, *args) == abi.GTP_E_RANGE
    assert lib.gtp_linear_wgrad_accum_bf16(MISALIGNED, ALIGNED, ALIGNED, 5, 10 ** 6, *args) == abi.GTP_E_ALIGN
    assert lib.gtp_linear_wgrad_accum_bf16(ALIGNED, ALIGNED, ALIGNED, 0, 10 ** 6, 256, 64, 64, abi.GTP_F32,
                                           None) == abi.GTP_E_DTYPE


def test_bf16_grad_sweep_argument_errors():
    lib = abi.load()
    h = abi.gtp_adam_hparams(3e-4, 0.9, 0.95, 1e-8, 0.1, 1, 1)
    ptrs = [ALIGNED + k * (1 << 24) for k in range(5)]   # distinct arrays (the sweep refuses overlaps)
    assert lib.gtp_adam_step_flat_bf16_grad(*ptrs, 100, None, None, 0, None, None) == abi.GTP_E_ARG
    assert lib.gtp_adam_step_flat_bf16_grad(MISALIGNED, *ptrs[1:], 100, None, None, 0, C.byref(h),
                                            None) == abi.GTP_E_ALIGN
    assert lib.gtp_adam_step_flat_bf16_grad(None, None, None, None, None, 0, None, None, 0, C.byref(h),
                                            None) == abi.GTP_OK


def test_columnwise_group_argument_errors_on_the_host():
    """Every descriptor is checked before a launch (no GPU needed for these)."""
    lib = abi.load()
    assert C.sizeof(abi.gtp_mx_col_desc) == 48
    d = (abi.gtp_mx_col_desc * 9)()
    assert lib.gtp_mxfp8_quantize_columnwise_group(d, 9, None) == abi.GTP_E_ARG      # more than eight
    assert lib.gtp_mxfp8_quantize_columnwise_group(d, -1, None) == abi.GTP_E_ARG
    assert lib.gtp_mxfp8_quantize_columnwise_group(None, 1, None) == abi.GTP_E_ARG
    assert lib.gtp_mxfp8_quantize_columnwise_group(d, 0, None) == abi.GTP_OK         # nothing to do
    assert lib.gtp_mxfp8_quantize_columnwise_group(d, 3, None) == abi.GTP_OK         # three empty matrices
    good = abi.gtp_mx_col_desc(ALIGNED, ALIGNED, ALIGNED, 64, 32, abi.GTP_F32, 0)
    cases = [(abi.gtp_mx_col_desc(ALIGNED, ALIGNED, ALIGNED, 64, 32, abi.GTP_F32, 2), abi.GTP_E_ARG),
             (abi.gtp_mx_col_desc(ALIGNED, ALIGNED, MISALIGNED, 64, 32, abi.GTP_F32, 1), abi.GTP_E_ALIGN),
             (abi.gtp_mx_col_desc(ALIGNED, ALIGNED, ALIGNED, 64, 32, abi.GTP_U8, 0), abi.GTP_E_DTYPE),
             (abi.gtp_mx_col_desc(ALIGNED, ALIGNED, ALIGNED, 48, 32, abi.GTP_F32, 0), abi.GTP_E_SHAPE),
             (abi.gtp_mx_col_desc(ALIGNED, MISALIGNED, ALIGNED, 64, 32, abi.GTP_F32, 0), abi.GTP_E_ALIGN),
             (abi.gtp_mx_col_desc(0x1002, ALIGNED, ALIGNED, 64, 32, abi.GTP_F32, 0), abi.GTP_E_ALIGN),
             (abi.gtp_mx_col_desc(None, ALIGNED, ALIGNED, 64, 32, abi.GTP_BF16, 0), abi.GTP_E_ARG)]
    for bad, status in cases:
        d[0], d[1] = good, bad     # the valid first matrix is not launched either
        assert lib.gtp_mxfp8_quantize_columnwise_group(d, 2, None) == status


def test_tiled_mxfp8_backward_argument_errors_on_the_host():
    lib = abi.load()
    u = (ALIGNED,) * 4
    # dgrad: dX rows of K = 64 bf16 (128 bytes); tiled scales must be 16-byte aligned
    assert lib.gtp_linear_dgrad_mxfp8_tiled(ALIGNED, MISALIGNED, ALIGNED, ALIGNED, ALIGNED, 256, 128, 64,
                                            None) == abi.GTP_E_ALIGN
    assert lib.gtp_linear_dgrad_mxfp8_tiled(*u, ALIGNED, 256, 100, 64, None) == abi.GTP_E_SHAPE   # N % 128
    assert lib.gtp_linear_wgrad_accum_mxfp8_tiled(ALIGNED, ALIGNED, ALIGNED, MISALIGNED, ALIGNED, 0, 10 ** 6,
                                                  256, 128, 64, None) == abi.GTP_E_ALIGN
    assert lib.gtp_linear_wgrad_accum_mxfp8_tiled(*u, ALIGNED, 0, 100, 256, 128, 64, None) == abi.GTP_E_RANGE
    assert lib.gtp_linear_wgrad_accum_mxfp8_tiled(*u, ALIGNED, 2, 10 ** 6, 256, 128, 64, None) == abi.GTP_E_ALIGN
    assert lib.gtp_mxfp8_quantize_columnwise_tiled(ALIGNED, abi.GTP_F32, 64, 32, ALIGNED, MISALIGNED,
                                                   None) == abi.GTP_E_ALIGN
    assert lib.gtp_mxfp8_quantize_columnwise_tiled(ALIGNED, abi.GTP_F32, 48, 32, ALIGNED, ALIGNED,
                                                   None) == abi.GTP_E_SHAPE


def test_rowwise_group_argument_errors_on_the_host():
    lib = abi.load()
    assert C.sizeof(abi.gtp_mx_row_desc) == 48
    d = (abi.gtp_mx_row_desc * 9)()
    assert lib.gtp_mxfp8_quantize_rowwise_group(d, 9, None) == abi.GTP_E_ARG
    assert lib.gtp_mxfp8_quantize_rowwise_group(None, 1, None) == abi.GTP_E_ARG
    assert lib.gtp_mxfp8_quantize_rowwise_group(d, 2, None) == abi.GTP_OK          # empty matrices
    good = abi.gtp_mx_row_desc(ALIGNED, ALIGNED, ALIGNED, 64, 32, abi.GTP_F32, 0)
    cases = [(abi.gtp_mx_row_desc(ALIGNED, ALIGNED, ALIGNED, 64, 32, abi.GTP_F32, 2), abi.GTP_E_ARG),
             (abi.gtp_mx_row_desc(ALIGNED, ALIGNED, ALIGNED, 64, 48, abi.GTP_F32, 0), abi.GTP_E_SHAPE),
             (abi.gtp_mx_row_desc(MISALIGNED, ALIGNED, ALIGNED, 64, 32, abi.GTP_BF16, 0), abi.GTP_E_ALIGN),
             (abi.gtp_mx_row_desc(ALIGNED, ALIGNED, ALIGNED, 64, 32, abi.GTP_U8, 1), abi.GTP_E_DTYPE)]
    for bad, status in cases:
        d[0], d[1] = good, bad     # the valid first matrix is not launched either
        assert lib.gtp_mxfp8_quantize_rowwise_group(d, 2, None) == status


def test_rs_local_sum_argument_errors_on_the_host():
    lib = abi.load()
    ptrs = lambda *p: (C.c_void_p * len(p))(*p)
    two = ptrs(ALIGNED, ALIGNED + 4096)
    assert lib.gtp_rs_local_sum(two, 0, 16, abi.GTP_BF16, ALIGNED + 8192, abi.GTP_BF16, None) == abi.GTP_E_ARG
    assert lib.gtp_rs_local_sum(two, 129, 16, abi.GTP_BF16, ALIGNED + 8192, abi.GTP_BF16, None) == abi.GTP_E_ARG
    assert lib.gtp_rs_local_sum(None, 2, 16, abi.GTP_BF16, ALIGNED + 8192, abi.GTP_BF16, None) == abi.GTP_E_ARG
    assert lib.gtp_rs_local_sum(two, 2, 16, abi.GTP_U8, ALIGNED + 8192, abi.GTP_BF16, None) == abi.GTP_E_DTYPE
    assert lib.gtp_rs_local_sum(two, 2, 0, abi.GTP_BF16, None, abi.GTP_BF16, None) == abi.GTP_OK      # empty
    assert lib.gtp_rs_local_sum(ptrs(ALIGNED, None), 2, 16, abi.GTP_BF16, ALIGNED + 8192, abi.GTP_BF16,
                                None) == abi.GTP_E_ARG
    assert lib.gtp_rs_local_sum(ptrs(ALIGNED, MISALIGNED), 2, 16, abi.GTP_BF16, ALIGNED + 8192, abi.GTP_BF16,
                                None) == abi.GTP_E_ALIGN
    assert lib.gtp_rs_local_sum(two, 2, 16, abi.GTP_BF16, MISALIGNED, abi.GTP_BF16, None) == abi.GTP_E_ALIGN
    # out overlapping a slice partly (16 bf16 elements = 32 bytes; out starts 16 bytes in)
    assert lib.gtp_rs_local_sum(two, 2, 16, abi.GTP_BF16, ALIGNED + 16, abi.GTP_BF16, None) == abi.GTP_E_ARG
    # out on a bf16 slice's start but fp32: not the same elements
    assert lib.gtp_rs_local_sum(two, 2, 16, abi.GTP_BF16, ALIGNED, abi.GTP_F32, None) == abi.GTP_E_ARG


def test_rs_local_sum_rows_argument_errors_on_the_host():
    lib = abi.load()
    f = lib.gtp_rs_local_sum_rows
    assert f(ALIGNED, 4096, 0, 16, abi.GTP_BF16, ALIGNED + (1 << 20), abi.GTP_BF16, None) == abi.GTP_E_ARG
    assert f(ALIGNED, 4096, 129, 16, abi.GTP_BF16, ALIGNED + (1 << 20), abi.GTP_BF16, None) == abi.GTP_E_ARG
    assert f(None, 4096, 2, 16, abi.GTP_BF16, ALIGNED + (1 << 20), abi.GTP_BF16, None) == abi.GTP_E_ARG
    assert f(ALIGNED, -32, 2, 16, abi.GTP_BF16, ALIGNED + (1 << 20), abi.GTP_BF16, None) == abi.GTP_E_ARG
    assert f(ALIGNED, 40, 2, 16, abi.GTP_BF16, ALIGNED + (1 << 20), abi.GTP_BF16, None) == abi.GTP_E_ALIGN  # row 1 at +40
    assert f(ALIGNED, 16, 2, 16, abi.GTP_BF16, ALIGNED + (1 << 20), abi.GTP_BF16, None) == abi.GTP_E_ARG    # rows overlap
    assert f(ALIGNED, 48, 2, 16, abi.GTP_F32, ALIGNED + (1 << 20), abi.GTP_F32, None) == abi.GTP_E_ARG      # 48 < 64
    assert f(ALIGNED, 4096, 2, 0, abi.GTP_BF16, None, abi.GTP_BF16, None) == abi.GTP_OK               # empty


def test_group_outputs_may_not_overlap_on_the_host():
    """A group whose outputs overlap a source or each other is refused before any launch
    (sources may be shared).  Distinct fake addresses 64 KiB apart; nothing launches."""
    lib = abi.load()
    a = [ALIGNED + k * 0x10000 for k in range(8)]
    R, Cc = 64, 32                                   # F32 source 8 KiB, codes 2 KiB, scales 64 B
    row = (abi.gtp_mx_row_desc * 2)()
    row[0] = abi.gtp_mx_row_desc(a[0], a[1], a[2], R, Cc, abi.GTP_F32, 0)
    row[1] = abi.gtp_mx_row_desc(a[3], a[1], a[4], R, Cc, abi.GTP_F32, 0)            # same codes as [0]
    assert lib.gtp_mxfp8_quantize_rowwise_group(row, 2, None) == abi.GTP_E_ARG
    row[1] = abi.gtp_mx_row_desc(a[3], a[4], a[3] + 4096, R, Cc, abi.GTP_F32, 0)     # scales inside its source
    assert lib.gtp_mxfp8_quantize_rowwise_group(row, 2, None) == abi.GTP_E_ARG
    row[1] = abi.gtp_mx_row_desc(a[3], a[0] + 16, a[4], R, Cc, abi.GTP_F32, 0)       # codes inside [0]'s source
    assert lib.gtp_mxfp8_quantize_rowwise_group(row, 2, None) == abi.GTP_E_ARG
    col = (abi.gtp_mx_col_desc * 2)()
    col[0] = abi.gtp_mx_col_desc(a[0], a[1], a[2], R, Cc, abi.GTP_F32, 0)
    col[1] = abi.gtp_mx_col_desc(a[3], a[4], a[1] + 1024, R, Cc, abi.GTP_F32, 0)     # scales inside [0]'s codes
    assert lib.gtp_mxfp8_quantize_columnwise_group(col, 2, None) == abi.GTP_E_ARG
    col[1] = abi.gtp_mx_col_desc(a[3], a[4], a[5], R, Cc, abi.GTP_F32, 1)            # tiled scales: 512 bytes
    col[0] = abi.gtp_mx_col_desc(a[0], a[5] + 256, a[2], R, Cc, abi.GTP_F32, 0)      # codes in them
    assert lib.gtp_mxfp8_quantize_columnwise_group(col, 2, None) == abi.GTP_E_ARG


def test_grouped_products_must_be_independent_on_the_host():
    """An output overlapping an input or another output is refused before any launch;
    shared inputs and overlapping fp32 wgrad views are not overlaps.  Fake addresses 16 MiB
    apart; the refused calls launch nothing."""
    lib = abi.load()
    a = [ALIGNED + k * (1 << 24) for k in range(8)]
    M, N, K = 256, 64, 64                                # bf16 [256, 64]: 32 KiB
    d = (abi.gtp_gemm_desc * 2)()
    d[0] = abi.gtp_gemm_desc(abi.GTP_GEMM_FPROP, abi.GTP_BF16, a[0], a[1], a[2], M, N, K, 0, 0)
    d[1] = abi.gtp_gemm_desc(abi.GTP_GEMM_DGRAD, abi.GTP_BF16, a[3], a[1], a[2] + 1024, M, N, K, 0, 0)
    assert lib.gtp_linear_grouped(d, 2, 0, None) == abi.GTP_E_ARG                 # two outputs overlap
    d[1] = abi.gtp_gemm_desc(abi.GTP_GEMM_DGRAD, abi.GTP_BF16, a[2], a[1], a[4], M, N, K, 0, 0)
    assert lib.gtp_linear_grouped(d, 2, 0, None) == abi.GTP_E_ARG                 # reads [0]'s output
    d[0] = abi.gtp_gemm_desc(abi.GTP_GEMM_FPROP, abi.GTP_BF16, a[0], a[1], a[0] + 64, M, N, K, 0, 0)
    assert lib.gtp_linear_grouped(d, 1, 0, None) == abi.GTP_E_ARG                 # output over its own input
    w = abi.gtp_gemm_desc(abi.GTP_GEMM_WGRAD_ACCUM, abi.GTP_BF16, a[5], a[6], a[7], M, N, K, 0, 10 ** 6)
    w.grad_dtype = abi.GTP_F32
    d[0] = abi.gtp_gemm_desc(abi.GTP_GEMM_DGRAD, abi.GTP_BF16, a[5], a[1], a[7] + 4096, M, N, K, 0, 0)
    d[1] = w
    assert lib.gtp_linear_grouped(d, 2, 0, None) == abi.GTP_E_ARG                 # dX inside the main_grad view


def test_sweep_arrays_may_not_overlap_on_the_host():
    """The fused sweep updates its arrays in place element by element: two arrays sharing a
    byte are refused before any launch.  Fake addresses; nothing launches."""
    lib = abi.load()
    h = abi.gtp_adam_hparams(3e-4, 0.9, 0.95, 1e-8, 0.1, 1, 1)
    a = [ALIGNED + k * (1 << 24) for k in range(6)]
    n = 1024
    assert lib.gtp_adam_step_flat(a[0], a[0], a[2], a[3], a[4], n, None, None, 0, C.byref(h), None) == abi.GTP_E_ARG
    assert b"overlaps" in lib.gtp_last_error()
    assert lib.gtp_adam_step_flat(a[0], a[1], a[2], a[3], a[2] + 2048, n, None, None, 0, C.byref(h),
                                  None) == abi.GTP_E_ARG                      # bf16 params inside exp_avg
    assert lib.gtp_adam_step_flat_bf16_grad(a[0], a[1], a[2], a[3], a[0] + 1024, n, None, None, 0, C.byref(h),
                                            None) == abi.GTP_E_ARG            # params inside the bf16 grads
    assert lib.gtp_adam_step_flat_mxfp8(a[0], a[1], a[2], a[3], a[4], a[4] + 512, n, None, None, 0, C.byref(h),
                                        None) == abi.GTP_E_ARG                # scales inside the codes
