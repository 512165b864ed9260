"""Empty and oversized inputs through the C ABI: every quantizer (each operand format,
both orientations and layouts) on tensors with no rows, no columns or
neither, the tensor scales and the statistics pass on no elements, and a
GEMM with no output rows or columns.  Each call returns SNIP_OK, writes
nothing outside its (empty) outputs -- guard bytes around them keep their
sentinel -- and still publishes what the oracle gives for an empty tensor:
amax 0, so g = s = 1 (the NVFP4 / FP8 scale definitions take 1 for an
all-zero tensor), and statistics sums and count 0.  The layer API has no
empty layer: T = 0 is SNIP_ERR_INVALID_ARG.  Dimensions beyond the kernels'
32-bit tile counts and TMA coordinates (above 2^31 - 1, or tensors of more
than 2^40 elements) are SNIP_ERR_SHAPE before anything is read or launched."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import need_gpu
from test_gpu_canary import Guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


SHAPES = [(0, 128), (128, 0), (0, 0)]


def _host_float(g):
    torch.cuda.synchronize()
    return float(np.frombuffer(g.buf[4096:4100].cpu().numpy().tobytes(), dtype=np.float32)[0])


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("orient", [0, 1])
@pytest.mark.parametrize("layout", [0, 1])
def test_quantizers_on_empty_tensors(snip, rows, cols, orient, layout):
    L = snip.load()
    src = torch.zeros(128, dtype=torch.bfloat16, device="cuda")   # a valid address that no call may read
    x = src.data_ptr() if rows * cols == 0 and (rows, cols) != (0, 0) else None
    ws = snip.small_workspace()
    st = torch.cuda.current_stream().cuda_stream
    orows, ocols = (rows, cols) if orient == 0 else (cols, rows)
    host = torch.zeros((rows, cols), dtype=torch.bfloat16)
    # NVFP4 (and its longer blocks), with per-block errors for the 16-element one
    for block in (16, 32, 64, 128):
        fmt = {16: snip.NVFP4, 32: snip.NVFP4_B32, 64: snip.NVFP4_B64, 128: snip.NVFP4_B128}[block]
        cb, sb = snip.snip_quantized_bytes(fmt, layout, orows, ocols)
        assert cb == 0 and sb == 0
        codes, scales, g = Guarded(0), Guarded(0), Guarded(4)
        if block == 16:
            err = Guarded(0)
            assert L.snip_quantize_nvfp4(x, rows, cols, orient, 1, 3, 5, None, layout, codes.ptr, scales.ptr, g.ptr,
                                         err.ptr, ws.ptr, ws.nbytes, st) == 0
            assert err.intact()
        else:
            assert L.snip_quantize_nvfp4_block(x, rows, cols, orient, 1, 3, 5, None, block, layout, codes.ptr,
                                               scales.ptr, g.ptr, ws.ptr, ws.nbytes, st) == 0
        assert codes.intact() and scales.intact()
        ref = oracle.quantize("nvfp4" if block == 16 else f"nvfp4-b{block}", host, orient, 1, 3, 5)
        assert _host_float(g) == float(ref.g) == 1.0
    # FP8 E4M3 and E5M2
    cb, _ = snip.snip_quantized_bytes(snip.FP8, layout, orows, ocols)
    assert cb == 0
    for fn, name in ((L.snip_quantize_fp8, "fp8"), (L.snip_quantize_e5m2, "e5m2")):
        codes, s = Guarded(0), Guarded(4)
        assert fn(x, rows, cols, orient, 1, 3, 6, None, layout, codes.ptr, s.ptr, ws.ptr, ws.nbytes, st) == 0
        assert codes.intact()
        assert _host_float(s) == float(oracle.quantize(name, host, orient, 1, 3, 6).s) == 1.0
    # MXFP4 (no tensor scale to publish)
    codes, scales = Guarded(0), Guarded(0)
    assert L.snip_quantize_mxfp4(x, rows, cols, orient, 1, 3, 7, layout, codes.ptr, scales.ptr, ws.ptr, ws.nbytes,
                                 st) == 0
    assert codes.intact() and scales.intact()
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK


def test_scales_and_statistics_of_no_elements(snip):
    L = snip.load()
    ws = snip.small_workspace()
    st = torch.cuda.current_stream().cuda_stream
    out = Guarded(12)
    assert L.snip_tensor_scales(None, 0, out.ptr, ws.ptr, ws.nbytes, st) == 0
    torch.cuda.synchronize()
    vals = np.frombuffer(out.buf[4096:4108].cpu().numpy().tobytes(), dtype=np.float32)
    assert list(vals) == [0.0, 1.0, 1.0] and out.intact()
    for rnd in (0, 1):
        for rows, cols in SHAPES:
            raw = Guarded(8 * snip.STATS_NVALS)
            b4, b8 = Guarded(0), Guarded(0)
            assert L.snip_quant_stats(None, rows, cols, rnd, 2, 9, None, raw.ptr, b4.ptr, b8.ptr, ws.ptr, ws.nbytes,
                                      st) == 0
            torch.cuda.synchronize()
            got = np.frombuffer(raw.buf[4096:4096 + 8 * snip.STATS_NVALS].cpu().numpy().tobytes(), dtype=np.float64)
            ref = oracle.quant_stats(torch.zeros((rows, cols), dtype=torch.bfloat16), rnd, 2, 9)["raw"]
            np.testing.assert_array_equal(got, ref)
            assert raw.intact() and b4.intact() and b8.intact()
    assert ws.status() == snip.SNIP_OK


@pytest.mark.parametrize("fmt", [1, 0])
def test_gemm_with_no_output(snip, fmt):
    L = snip.load()
    K = 256
    a = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    ws = snip.small_workspace()
    st = torch.cuda.current_stream().cuda_stream
    for M, N in ((0, 256), (256, 0), (0, 0)):
        D = Guarded(0)
        s = sc.data_ptr() if fmt == 1 else None
        assert L.snip_gemm(fmt, a.data_ptr(), s, g.data_ptr(), a.data_ptr(), s, g.data_ptr(), M, N, K, D.ptr,
                           max(N, 4), ws.ptr, ws.nbytes, st) == 0
        assert D.intact()
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK


def test_layer_without_tokens_is_rejected(snip):
    plan = snip.Plan([snip.NVFP4, snip.FP8])
    L = snip.load()
    X = torch.zeros((16, 128), dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros((16, 128), dtype=torch.float32, device="cuda")
    ws = snip.Workspace(1 << 20)
    for layer in (0, 1):
        assert L.snip_qlinear_workspace_size(plan.handle, layer, 0, 128, 128) == 0
        assert L.snip_qlinear_fwd(plan.handle, layer, X.data_ptr(), X.data_ptr(), 0, 128, 128, Y.data_ptr(), None,
                                  ws.ptr, ws.nbytes, torch.cuda.current_stream().cuda_stream) == \
            snip.SNIP_ERR_INVALID_ARG


def test_oversized_dimensions_rejected(snip):
    L = snip.load()
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")   # never read: the size checks come first
    P = buf.data_ptr()
    ws = snip.small_workspace()
    st = torch.cuda.current_stream().cuda_stream
    big, wide = 1 << 31, 1 << 26                         # 2^31 rows; 2^26 x 2^26 = 2^52 elements
    for rows, cols in ((big, 16), (16, big), (wide, wide)):
        assert L.snip_quantize_nvfp4(P, rows, cols, 0, 0, 0, 0, None, 0, P, P, P, None, ws.ptr, ws.nbytes,
                                     st) == snip.SNIP_ERR_SHAPE
        assert L.snip_quantize_fp8(P, rows, cols, 1, 0, 0, 0, None, 1, P, P, ws.ptr, ws.nbytes,
                                   st) == snip.SNIP_ERR_SHAPE
        assert L.snip_quant_stats(P, rows, cols, 0, 0, 0, None, P, None, None, ws.ptr, ws.nbytes,
                                  st) == snip.SNIP_ERR_SHAPE
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    for M, N, K in ((big, 256, 256), (256, big, 256), (256, 256, big), (wide, wide, 256)):
        assert L.snip_gemm(1, P, P, g.data_ptr(), P, P, g.data_ptr(), M, N, K, P, N, ws.ptr, ws.nbytes,
                           st) == snip.SNIP_ERR_SHAPE
    plan = snip.Plan([snip.NVFP4])
    for T, K, N in ((big, 256, 256), (256, big, 256), (wide, wide, 256)):
        assert L.snip_qlinear_workspace_size(plan.handle, 0, T, K, N) == 0
        assert L.snip_qlinear_fwd(plan.handle, 0, P, P, T, K, N, P, None, ws.ptr, ws.nbytes, st) == \
            snip.SNIP_ERR_SHAPE
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK
