"""Degenerate GEMM shapes through snip_gemm, for every operand format: one-row
and one-column outputs, the shortest contraction (one 16-element block; 32
for MXFP4) and contractions that fill no whole 256-element stage, row and
column counts off every tile boundary.  D sits inside a wider row pitch
(the pitch is a multiple of 4 elements, so a one-column D has pitch 4).
D matches the oracle's fp64 product of the dequantized operands within the
GEMM bounds, and the pitch padding keeps its sentinel."""
import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import gemm_close, need_gpu

pytestmark = pytest.mark.gpu

SENTINEL = 7.0e30


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


SHAPES = [(1, 1, 16), (1, 300, 48), (17, 1, 272), (255, 257, 16), (257, 33, 4096), (33, 511, 1040)]


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8", "mxfp4"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_degenerate_shapes(snip, fmt, M, N, K):
    if fmt == "mxfp4":
        K = (K + 31) // 32 * 32          # MXFP4 blocks are 32 elements
    A = inputs.normal_bf16((M, K), 1.0, 90 + M, 1)
    B = inputs.normal_bf16((N, K), 0.02, 90 + N, 2)
    quant = {"nvfp4": snip.quantize_nvfp4, "fp8": snip.quantize_fp8, "mxfp4": snip.quantize_mxfp4}[fmt]
    code = {"nvfp4": snip.NVFP4, "fp8": snip.FP8, "mxfp4": snip.MXFP4}[fmt]
    a = quant(A.cuda(), rnd=1, seed=4, stream_id=2, layout=snip.MMA)
    b = quant(B.cuda(), rnd=1, seed=4, stream_id=3, layout=snip.MMA)
    ldd = (N + 3) // 4 * 4 + 4
    big = torch.full((M, ldd), SENTINEL, dtype=torch.float32, device="cuda")
    D = big[:, :N]
    ws = snip.small_workspace()
    snip.gemm(code, a, b, M, N, K, out=D, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK
    ref = oracle.gemm_tn(oracle.quantize(fmt, A, 0, 1, 4, 2).dequant(), oracle.quantize(fmt, B, 0, 1, 4, 3).dequant())
    gemm_close(D.cpu().numpy(), ref, f"{fmt} {M}x{N}x{K}")
    assert np.all(big[:, N:].cpu().numpy() == SENTINEL), "pitch padding written"
