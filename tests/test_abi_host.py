"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every symbol include/snip.h declares, and its host-only
entry points (status text, layout sizes, plans, statistics finalisation)
behave as documented.  No kernel is launched."""
import math
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def snip():
    from sub_byte_mixed_gb300 import build, snip as s
    build.build()
    s.load()
    return s


def _declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "snip.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(snip_[a-z0-9_]+)\s*\(", hdr)))


def test_every_declared_symbol_is_exported(snip):
    lib = snip.load()
    declared = _declared_symbols()
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(snip.EXPORTS) == declared


def test_status_strings(snip):
    for code in range(9):
        assert snip.status_string(code)
    assert "aligned" in snip.status_string(snip.SNIP_ERR_ALIGN)


def test_quantized_bytes(snip):
    assert snip.snip_quantized_bytes(snip.NVFP4, snip.ROWMAJOR, 64, 128) == (64 * 64, 64 * 8)
    assert snip.snip_quantized_bytes(snip.FP8, snip.ROWMAJOR, 64, 128) == (64 * 128, 0)
    # MMA layout: rows padded to 256, contraction to 256 (NVFP4) / 128 (FP8)
    assert snip.snip_quantized_bytes(snip.NVFP4, snip.MMA, 64, 128) == (256 * 128, 256 * 16)
    assert snip.snip_quantized_bytes(snip.FP8, snip.MMA, 300, 130) == (512 * 256, 0)
    # MXFP4: NVFP4's codes, one E8M0 byte per 32 elements
    assert snip.snip_quantized_bytes(snip.MXFP4, snip.ROWMAJOR, 64, 128) == (64 * 64, 64 * 4)
    assert snip.snip_quantized_bytes(snip.MXFP4, snip.MMA, 64, 288) == (256 * 256, 256 * 16)
    # longer NVFP4 blocks use NVFP4's layouts (one scale byte per 16 elements)
    for f in (snip.NVFP4_B32, snip.NVFP4_B64, snip.NVFP4_B128):
        for layout, r, c in ((snip.ROWMAJOR, 64, 256), (snip.MMA, 300, 384)):
            assert snip.snip_quantized_bytes(f, layout, r, c) == snip.snip_quantized_bytes(snip.NVFP4, layout, r, c)
    for bad in (snip.FP8_E5M2_GRAD, 8, -1):   # a layer-only format, then no format
        with pytest.raises(snip.SnipError):
            snip.snip_quantized_bytes(bad, 0, 1, 1)


def test_plan_and_workspace_sizes(snip):
    plan = snip.Plan([snip.NVFP4, snip.FP8, snip.NVFP4], seed=7)
    import ctypes
    f, sd = ctypes.c_int(), ctypes.c_uint64()
    assert snip.load().snip_plan_get(plan.handle, 1, ctypes.byref(f), ctypes.byref(sd)) == 0
    assert f.value == snip.FP8 and sd.value == 7
    assert snip.load().snip_plan_get(plan.handle, 3, None, None) == snip.SNIP_ERR_INVALID_ARG
    with pytest.raises(snip.SnipError):
        plan.set_rounding(0, 6, snip.RTN)
    plan.set_rounding(0, snip.TAG_WT_DGRAD, snip.RTN)
    ws4 = snip.snip_qlinear_workspace_size(plan.handle, 0, 64, 128, 128)
    ws8 = snip.snip_qlinear_workspace_size(plan.handle, 1, 64, 128, 128)
    assert ws4 > 0 and ws8 > 0
    # backward operands dominate: dY (T,N), W^T (K,N), dY^T (N,T), X^T (K,T), each padded
    b = sum(sum(snip.snip_quantized_bytes(snip.NVFP4, snip.MMA, r, c)) for r, c in
            [(64, 128), (128, 128), (128, 64), (128, 64)])
    assert ws4 >= b
    assert snip.snip_qlinear_workspace_size(plan.handle, 0, 64, 120, 128) == 0     # K % 16 != 0
    with pytest.raises(snip.SnipError):
        snip.Plan([snip.NVFP4, 9])


def test_stats_finalize_flags(snip):
    raw = [3.0003, 1.0, 1.0002, 0.5, 0.1, 2.0, 16.0, 0.0]
    st = snip.snip_stats_finalize(raw)
    assert st.ratio_nvfp4 == pytest.approx(math.sqrt(3.0003))
    assert st.below_sqrt3_nvfp4 == 0 and st.below_sqrt3_fp8 == 1
    z = snip.snip_stats_finalize([0.0] * 8)
    assert math.isinf(z.ratio_nvfp4) and z.below_sqrt3_nvfp4 == 0


def test_calls_without_usable_gpu_fail_loudly(snip):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert snip.load().snip_device_check() in (snip.SNIP_ERR_CUDA, snip.SNIP_ERR_UNSUPPORTED_DEVICE)
    st = snip.load().snip_amax(16, 8, 16, 16, 1 << 20, None)
    assert st in (snip.SNIP_ERR_CUDA, snip.SNIP_ERR_UNSUPPORTED_DEVICE)


def test_library_reports_the_header_version():
    """snip_version() (no device needed) matches SNIP_ABI_VERSION in include/snip.h."""
    import re
    from sub_byte_mixed_gb300 import snip
    hdr = open(os.path.join(ROOT, "include", "snip.h")).read()
    want = int(re.search(r"#define SNIP_ABI_VERSION (\d+)", hdr).group(1))
    assert snip.load().snip_version() == want


def test_quantize_part_index_rules_need_no_device(snip):
    """snip_quantize_part checks where the part starts before it touches the
    device: the part begins on a whole row (index_base a multiple of cols and
    of 16), and with blocks along the rows (the tokens) on a whole block of
    rows, so no block straddles two parts.  Pointers are dummies: a call that
    passes these rules goes on to the device check (which fails on a host
    without a usable GPU, and would reject the dummies' alignment on one)."""
    lib = snip.load()
    P = 4096   # dummy, 16-byte aligned, never dereferenced by a rejected call

    def part(fmt, orient, rows, cols, index_base):
        return lib.snip_quantize_part(fmt, P, rows, cols, orient, snip.SR, 0, 0, index_base, P, snip.ROWMAJOR,
                                      P, P, None, P, 1 << 20, None)

    C = 256
    # along the rows: the first row must be a whole number of blocks (16 for NVFP4, 32 for MXFP4)
    assert part(snip.NVFP4, snip.ALONG_ROWS, 64, C, 8 * C) == snip.SNIP_ERR_SHAPE
    assert part(snip.MXFP4, snip.ALONG_ROWS, 64, C, 16 * C) == snip.SNIP_ERR_SHAPE
    assert part(snip.FP8, snip.ALONG_ROWS, 64, C, 24 * C) == snip.SNIP_ERR_SHAPE
    # not a whole row, or not a multiple of 16
    assert part(snip.NVFP4, snip.ALONG_COLS, 64, C, 16) == snip.SNIP_ERR_SHAPE
    assert part(snip.NVFP4, snip.ALONG_COLS, 64, 48, 8) == snip.SNIP_ERR_SHAPE
    # bad orientation
    assert part(snip.NVFP4, 7, 64, C, 0) == snip.SNIP_ERR_INVALID_ARG
    import torch
    if torch.cuda.is_available():
        return
    # valid starts reach the device check
    for fmt, orient, first_row in ((snip.NVFP4, snip.ALONG_ROWS, 16), (snip.MXFP4, snip.ALONG_ROWS, 32),
                                   (snip.NVFP4, snip.ALONG_COLS, 3), (snip.FP8, snip.ALONG_ROWS, 48)):
        st = part(fmt, orient, 64, C, first_row * C)
        assert st in (snip.SNIP_ERR_CUDA, snip.SNIP_ERR_UNSUPPORTED_DEVICE), (fmt, orient, st)
