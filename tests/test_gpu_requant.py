"""NEXT-3: the GEMM whose product feeds the next layer writes it quantized
(NVFP4 row blocks of bf16(D), given tensor scale).  Checked three ways:
bit-exact against the library's own quantizer applied to bf16 of the D it
returns (the definition of the fused path; that quantizer is bit-exact
against the oracle elsewhere); against the oracle's quantization of its fp64
product rounded to bf16 -- codes may differ only where fp32 and fp64
accumulation round to different bf16 values, so nearly all must agree and
every difference is a neighbouring grid value; and the amax output exactly."""
import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import mma_codes_to_rowmajor, mma_scales_to_rowmajor, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


def _mag(codes):
    lo, hi = codes & 0x0F, codes >> 4
    return np.stack([lo & 7, hi & 7], -1).reshape(codes.shape[0], -1)


@pytest.mark.parametrize("fmt", [1, 0])
@pytest.mark.parametrize("M,N,K", [(192, 160, 256), (272, 400, 336), (2048, 2560, 512)])
@pytest.mark.parametrize("rnd", [0, 1])
def test_requant_product(snip, fmt, M, N, K, rnd):
    A = inputs.normal_bf16((M, K), 1e-3, 12, 1)       # a gradient-like operand (dY)
    B = inputs.normal_bf16((N, K), 0.02, 12, 2)       # and a weight-like one (W^T)
    q = snip.quantize_nvfp4 if fmt == 1 else snip.quantize_fp8
    a = q(A.cuda(), rnd=1, seed=1, stream_id=2, layout=snip.MMA)
    b = q(B.cuda(), rnd=1, seed=1, stream_id=3, layout=snip.MMA)
    # a delayed tensor scale: the product's amax estimated at 80% of its true value, so some values saturate
    fname = "nvfp4" if fmt == 1 else "fp8"
    ref = oracle.gemm_tn(oracle.quantize(fname, A, 0, 1, 1, 2).dequant(), oracle.quantize(fname, B, 0, 1, 1, 3).dequant())
    g = torch.tensor([0.8 * float(np.abs(ref).max()) / 2688.0], dtype=torch.float32, device="cuda")
    D, rq, amax = snip.gemm_requant(fmt, a, b, M, N, K, g, rnd=rnd, seed=7, stream_id=11)
    torch.cuda.synchronize()
    # 1. bit-exact against quantizing bf16(D) with the same scale, rounding and random bits
    Db = D.to(torch.bfloat16)
    ref_gpu = snip.quantize_nvfp4(Db, rnd=rnd, seed=7, stream_id=11, g_in=g, layout=snip.MMA)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(rq.codes.cpu().numpy(), ref_gpu.codes.cpu().numpy())
    np.testing.assert_array_equal(rq.scales.cpu().numpy(), ref_gpu.scales.cpu().numpy())
    assert float(amax.cpu()) == float(Db.float().abs().max())
    # 2. against the oracle: its fp64 product rounded to bf16, quantized
    orc = oracle.quantize_nvfp4(torch.from_numpy(ref).to(torch.bfloat16), rnd=rnd, seed=7, stream_id=11,
                                g_in=float(g.cpu()))
    _, codes = mma_codes_to_rowmajor(rq.codes, M, N, fmt_nvfp4=True)
    _, scales = mma_scales_to_rowmajor(rq.scales, M, N)
    assert np.mean(scales == orc.scales) > 0.999
    same = codes == orc.codes
    assert np.mean(same) > 0.999
    mg, mo = _mag(codes), _mag(orc.codes)
    assert np.all(np.abs(mg.astype(int) - mo.astype(int)) <= 1)
    assert float(amax.cpu()) == pytest.approx(float(np.abs(ref).max()), rel=2 ** -7)


def test_requant_without_fp32_output(snip):
    M, N, K = 256, 512, 256
    A = inputs.normal_bf16((M, K), 1.0, 13, 1)
    B = inputs.normal_bf16((N, K), 0.02, 13, 2)
    a = snip.quantize_nvfp4(A.cuda(), layout=snip.MMA)
    b = snip.quantize_nvfp4(B.cuda(), layout=snip.MMA)
    g = torch.tensor([1e-3], dtype=torch.float32, device="cuda")
    D, rq1, _ = snip.gemm_requant(snip.NVFP4, a, b, M, N, K, g, rnd=1, seed=3, stream_id=4)
    none, rq2, _ = snip.gemm_requant(snip.NVFP4, a, b, M, N, K, g, rnd=1, seed=3, stream_id=4, want_d=False)
    torch.cuda.synchronize()
    assert none is None
    np.testing.assert_array_equal(rq1.codes.cpu().numpy(), rq2.codes.cpu().numpy())
    np.testing.assert_array_equal(rq1.scales.cpu().numpy(), rq2.scales.cpu().numpy())
    # the re-quantized operand feeds the next GEMM like any quantizer output
    C = inputs.normal_bf16((128, N), 0.02, 13, 3)
    c = snip.quantize_nvfp4(C.cuda(), layout=snip.MMA)
    out = snip.gemm(snip.NVFP4, rq2, c, M, 128, N)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
