"""The CTA-pair GEMM's output path: each epilogue warp stages 32 x 32 fp32
boxes of D in shared memory and writes them with TMA stores, which leave
out every element past M or N.  Checked on ragged shapes large enough for
the pair kernel (at least one 256 x 256 tile per SM pair), for every operand
format, with D inside a wider row pitch: D matches the oracle's product
within the GEMM bounds, the pitch's padding columns and the rows around D
keep their sentinel, so no box writes outside M x N."""
import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import gemm_close, need_gpu

pytestmark = pytest.mark.gpu

SENTINEL = -12345.0


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


def _quantized(snip, fmt, X, sid):
    if fmt == "nvfp4":
        return snip.quantize_nvfp4(X.cuda(), stream_id=sid, layout=snip.MMA)
    if fmt == "mxfp4":
        return snip.quantize_mxfp4(X.cuda(), stream_id=sid, layout=snip.MMA)
    return snip.quantize_fp8(X.cuda(), stream_id=sid, layout=snip.MMA)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "fp8"])
@pytest.mark.parametrize("M,N,ldd_pad", [(2000, 2600, 0), (2000, 2600, 60), (2304, 2832, 4)])
def test_pair_gemm_ragged_output(snip, fmt, M, N, ldd_pad):
    K = 512
    assert ((M + 255) // 256) * ((N + 255) // 256) >= 76   # the pair kernel on a 152-SM GB300
    A = inputs.normal_bf16((M, K), 1.0, 41, 1)
    B = inputs.normal_bf16((N, K), 0.02, 41, 2)
    a = _quantized(snip, fmt, A, 2)
    b = _quantized(snip, fmt, B, 3)
    ldd = N + ldd_pad
    big = torch.full((M + 64, ldd), SENTINEL, dtype=torch.float32, device="cuda")   # 32 guard rows each side
    D = big[32:32 + M, :N]
    code = {"nvfp4": snip.NVFP4, "mxfp4": snip.MXFP4, "fp8": snip.FP8}[fmt]
    ws = snip.small_workspace()
    snip.gemm(code, a, b, M, N, K, out=D, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK
    ref = oracle.gemm_tn(oracle.quantize(fmt, A, 0, 0, 0, 2).dequant(), oracle.quantize(fmt, B, 0, 0, 0, 3).dequant())
    gemm_close(D.cpu().numpy(), ref, f"{fmt} {M}x{N} ldd {ldd}")
    h = big.cpu().numpy()
    assert np.all(h[:32] == SENTINEL) and np.all(h[32 + M:] == SENTINEL), "rows outside D written"
    if ldd_pad:
        assert np.all(h[32:32 + M, N:] == SENTINEL), "pitch padding written"
