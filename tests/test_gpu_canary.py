"""Guard bytes around every output buffer: each output of the quantizers
(both layouts and orientations, every operand format, with per-block errors),
the statistics (raw sums and per-block errors, standalone and fused), the
shard quantizer and the GEMM is written into the middle of a larger buffer
whose 4 KB on either side hold a sentinel byte; after the call the sentinels
must be untouched, so no kernel writes before or past the buffer sizes the
C ABI documents (snip_quantized_bytes, rows x blocks for errors, 8 doubles of
statistics, M x ldd for D).  Shapes are ragged (272 x 400: neither a multiple
of the 256-row MMA padding nor of a 32-block segment)."""
import pytest
import torch

from sub_byte_mixed_gb300 import inputs
from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu

PAD = 4096
SENTINEL = 0xA5


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


class Guarded:
    """nbytes usable device bytes, 16-byte aligned, with PAD sentinel bytes on each side."""

    def __init__(self, nbytes):
        self.n = max(int(nbytes), 0)
        self.buf = torch.full((self.n + 2 * PAD,), SENTINEL, dtype=torch.uint8, device="cuda")

    @property
    def ptr(self):
        return self.buf.data_ptr() + PAD

    def intact(self):
        torch.cuda.synchronize()
        head = self.buf[:PAD]
        tail = self.buf[PAD + self.n:]
        return bool((head == SENTINEL).all()) and bool((tail == SENTINEL).all())


def _check(*bufs):
    for i, b in enumerate(bufs):
        assert b.intact(), f"output {i} ({b.n} bytes) written outside its bounds"


R, C = 272, 400


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("orient", [0, 1])
@pytest.mark.parametrize("rnd", [0, 1])
def test_quantizers_stay_in_bounds(snip, layout, orient, rnd):
    L = snip.load()
    x = inputs.outlier_bf16(R, C, seed=3, tensor_id=9).cuda()
    ws = snip.small_workspace()
    st = torch.cuda.current_stream().cuda_stream
    orows, ocols = (R, C) if orient == 0 else (C, R)
    # NVFP4 with per-block errors
    cb, sb = snip.snip_quantized_bytes(snip.NVFP4, layout, orows, ocols)
    codes, scales, g, err = Guarded(cb), Guarded(sb), Guarded(4), Guarded(orows * (ocols // 16) * 4)
    assert L.snip_quantize_nvfp4(x.data_ptr(), R, C, orient, rnd, 1, 2, None, layout, codes.ptr, scales.ptr, g.ptr,
                                 err.ptr, ws.ptr, ws.nbytes, st) == 0
    _check(codes, scales, g, err)
    # FP8 E4M3 and E5M2
    cb, _ = snip.snip_quantized_bytes(snip.FP8, layout, orows, ocols)
    codes, s = Guarded(cb), Guarded(4)
    assert L.snip_quantize_fp8(x.data_ptr(), R, C, orient, rnd, 1, 3, None, layout, codes.ptr, s.ptr, ws.ptr,
                               ws.nbytes, st) == 0
    _check(codes, s)
    codes, s = Guarded(cb), Guarded(4)
    assert L.snip_quantize_e5m2(x.data_ptr(), R, C, orient, rnd, 1, 4, None, layout, codes.ptr, s.ptr, ws.ptr,
                                ws.nbytes, st) == 0
    _check(codes, s)
    # MXFP4 (32-element blocks) and NVFP4 with 32-element blocks need the blocked dim % 32
    x32 = inputs.outlier_bf16(288, 416, seed=3, tensor_id=10).cuda()
    o32 = (288, 416) if orient == 0 else (416, 288)
    cb, sb = snip.snip_quantized_bytes(snip.MXFP4, layout, *o32)
    codes, scales = Guarded(cb), Guarded(sb)
    assert L.snip_quantize_mxfp4(x32.data_ptr(), 288, 416, orient, rnd, 1, 5, layout, codes.ptr, scales.ptr, ws.ptr,
                                 ws.nbytes, st) == 0
    _check(codes, scales)
    cb, sb = snip.snip_quantized_bytes(snip.NVFP4_B32, layout, *o32)
    codes, scales, g = Guarded(cb), Guarded(sb), Guarded(4)
    assert L.snip_quantize_nvfp4_block(x32.data_ptr(), 288, 416, orient, rnd, 1, 6, None, 32, layout, codes.ptr,
                                       scales.ptr, g.ptr, ws.ptr, ws.nbytes, st) == 0
    _check(codes, scales, g)
    assert ws.status() == snip.SNIP_OK


@pytest.mark.parametrize("rnd", [0, 1])
def test_statistics_stay_in_bounds(snip, rnd):
    L = snip.load()
    x = inputs.outlier_bf16(R, C, seed=4, tensor_id=9).cuda()
    ws = snip.small_workspace()
    st = torch.cuda.current_stream().cuda_stream
    raw, b4, b8 = Guarded(8 * snip.STATS_NVALS), Guarded(R * (C // 16) * 4), Guarded(R * (C // 16) * 4)
    assert L.snip_quant_stats(x.data_ptr(), R, C, rnd, 2, 7, None, raw.ptr, b4.ptr, b8.ptr, ws.ptr, ws.nbytes,
                              st) == 0
    _check(raw, b4, b8)
    for fmt in (snip.NVFP4, snip.FP8, snip.MXFP4, snip.FP8_E5M2):
        cols = 416 if fmt == snip.MXFP4 else C
        xf = inputs.outlier_bf16(R, cols, seed=4, tensor_id=11).cuda()
        for layout in (0, 1):
            cb, sb = snip.snip_quantized_bytes(fmt, layout, R, cols)
            codes, scales, raw = Guarded(cb), Guarded(max(sb, 0)), Guarded(8 * snip.STATS_NVALS)
            assert L.snip_quantize_stats(fmt, xf.data_ptr(), R, cols, rnd, 2, 8, None, layout, codes.ptr,
                                         scales.ptr if sb else None, raw.ptr, ws.ptr, ws.nbytes, st) == 0
            _check(codes, scales, raw)
    assert ws.status() == snip.SNIP_OK


@pytest.mark.parametrize("orient", [0, 1])
def test_shard_quantizer_stays_in_bounds(snip, orient):
    L = snip.load()
    x = inputs.normal_bf16((256, C), 1.0, 5, 2).cuda()
    sc = snip.tensor_scales(x)
    ws = snip.small_workspace()
    st = torch.cuda.current_stream().cuda_stream
    part = x[128:].contiguous()
    orows, ocols = (128, C) if orient == 0 else (C, 128)
    for layout in (0, 1):
        cb, sb = snip.snip_quantized_bytes(snip.NVFP4, layout, orows, ocols)
        codes, scales = Guarded(cb), Guarded(sb)
        raw = Guarded(8 * snip.STATS_NVALS) if orient == 0 else None
        assert L.snip_quantize_part(snip.NVFP4, part.data_ptr(), 128, C, orient, 1, 3, 9, 128 * C, sc.data_ptr(),
                                    layout, codes.ptr, scales.ptr, raw.ptr if raw else None, ws.ptr, ws.nbytes,
                                    st) == 0
        _check(codes, scales, *([raw] if raw else []))
    assert ws.status() == snip.SNIP_OK


@pytest.mark.parametrize("fmt", [1, 0])
def test_gemm_output_stays_in_bounds(snip, fmt):
    M, N, K = 272, 400, 336
    A = inputs.normal_bf16((M, K), 1.0, 6, 1).cuda()
    B = inputs.normal_bf16((N, K), 0.02, 6, 2).cuda()
    q = snip.quantize_nvfp4 if fmt == 1 else snip.quantize_fp8
    a = q(A, layout=snip.MMA)
    b = q(B, layout=snip.MMA)
    D = Guarded(M * N * 4)
    ws = snip.small_workspace()
    L = snip.load()
    sa = a.scales.data_ptr() if fmt == 1 else None
    sb = b.scales.data_ptr() if fmt == 1 else None
    ga = (a.g if fmt == 1 else a.s).data_ptr()
    gb = (b.g if fmt == 1 else b.s).data_ptr()
    assert L.snip_gemm(fmt, a.codes.data_ptr(), sa, ga, b.codes.data_ptr(), sb, gb, M, N, K, D.ptr, N, ws.ptr,
                       ws.nbytes, torch.cuda.current_stream().cuda_stream) == 0
    _check(D)
    assert ws.status() == snip.SNIP_OK
