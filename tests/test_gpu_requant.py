"""NEXT-3: the GEMM whose product feeds the next layer writes it quantized
(NVFP4 row and column blocks of bf16(D), given tensor scale).  Checked:
bit-exact against the oracle on operands whose products are exact in fp32
(every partial sum representable, power-of-two tensor scales), where the
GPU's fp32 product must equal the oracle's fp64 one and the oracle's
quantization of its own bf16(product) fixes every code and scale; on general
operands, bit-exact against the library's own quantizer applied to bf16 of
the D it returns (the definition of the fused path; that quantizer is
bit-exact against the oracle elsewhere) and, against the oracle, codes equal
except where fp32 and fp64 accumulation round to different bf16 values (only
to a neighbouring grid value); and the amax output exactly."""
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
    D, rq, amax, _ = snip.gemm_requant(fmt, a, b, M, N, K, g, rnd=rnd, seed=7, stream_id=11)
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
    D, rq1, _, _ = snip.gemm_requant(snip.NVFP4, a, b, M, N, K, g, rnd=1, seed=3, stream_id=4)
    none, rq2, _, _ = snip.gemm_requant(snip.NVFP4, a, b, M, N, K, g, rnd=1, seed=3, stream_id=4, want_d=False)
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


# ---------------------------------------------------------------- column blocks (the transposed operand)

def _operands(snip, fmt, M, N, K, seed):
    A = inputs.normal_bf16((M, K), 1e-3, seed, 1)
    B = inputs.normal_bf16((N, K), 0.02, seed, 2)
    q = snip.quantize_nvfp4 if fmt == 1 else snip.quantize_fp8
    a = q(A.cuda(), rnd=1, seed=1, stream_id=2, layout=snip.MMA)
    b = q(B.cuda(), rnd=1, seed=1, stream_id=3, layout=snip.MMA)
    fname = "nvfp4" if fmt == 1 else "fp8"
    ref = oracle.gemm_tn(oracle.quantize(fname, A, 0, 1, 1, 2).dequant(), oracle.quantize(fname, B, 0, 1, 1, 3).dequant())
    return a, b, ref


# (192, 160) and (272, 400): one-CTA tiles, M not a multiple of 256 (272 also leaves 128 rows of the
# 256-row padding uncovered); (2048, 2560): CTA-pair tiles
@pytest.mark.parametrize("fmt", [1, 0])
@pytest.mark.parametrize("M,N,K", [(192, 160, 256), (272, 400, 336), (2048, 2560, 512)])
@pytest.mark.parametrize("rnd,rnd_t", [(0, 0), (1, 1), (0, 1)])
def test_requant_both_orientations(snip, fmt, M, N, K, rnd, rnd_t):
    a, b, ref = _operands(snip, fmt, M, N, K, 14)
    g = torch.tensor([0.8 * float(np.abs(ref).max()) / 2688.0], dtype=torch.float32, device="cuda")
    D, rq, amax, rq_t = snip.gemm_requant(fmt, a, b, M, N, K, g, rnd=rnd, seed=9, stream_id=21, cols=True,
                                          rnd_t=rnd_t, stream_id_t=23)
    torch.cuda.synchronize()
    Db = D.to(torch.bfloat16)
    # 1. bit-exact: each orientation equals the library quantizer on bf16(D), same scale, rounding, bits
    ref_r = snip.quantize_nvfp4(Db, rnd=rnd, seed=9, stream_id=21, g_in=g, layout=snip.MMA)
    ref_c = snip.quantize_nvfp4(Db, orient=snip.ALONG_ROWS, rnd=rnd_t, seed=9, stream_id=23, g_in=g, layout=snip.MMA)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(rq.codes.cpu().numpy(), ref_r.codes.cpu().numpy())
    np.testing.assert_array_equal(rq.scales.cpu().numpy(), ref_r.scales.cpu().numpy())
    assert rq_t.codes.numel() == ref_c.codes.numel() and rq_t.scales.numel() == ref_c.scales.numel()
    np.testing.assert_array_equal(rq_t.codes.cpu().numpy(), ref_c.codes.cpu().numpy())
    np.testing.assert_array_equal(rq_t.scales.cpu().numpy(), ref_c.scales.cpu().numpy())
    assert float(amax.cpu()) == float(Db.float().abs().max())
    # 2. the column blocks against the oracle's transposed quantization of its fp64 product in bf16
    orc = oracle.quantize_nvfp4(torch.from_numpy(ref).to(torch.bfloat16), orient=1, rnd=rnd_t, seed=9, stream_id=23,
                                g_in=float(g.cpu()))
    _, codes = mma_codes_to_rowmajor(rq_t.codes, N, M, fmt_nvfp4=True)
    _, scales = mma_scales_to_rowmajor(rq_t.scales, N, M)
    assert np.mean(scales == orc.scales) > 0.999
    assert np.mean(codes == orc.codes) > 0.999
    mg, mo = _mag(codes), _mag(orc.codes)
    assert np.all(np.abs(mg.astype(int) - mo.astype(int)) <= 1)


def test_requant_columns_only_and_as_wgrad_operand(snip):
    """Column blocks alone equal those written beside the row blocks, and feed the next GEMM (the
    preceding layer's wgrad, contraction over the tokens M) exactly like the quantizer's output."""
    M, N, K = 512, 256, 256
    a, b, ref = _operands(snip, 1, M, N, K, 15)
    g = torch.tensor([float(np.abs(ref).max()) / 2688.0], dtype=torch.float32, device="cuda")
    _, _, _, both = snip.gemm_requant(snip.NVFP4, a, b, M, N, K, g, rnd=1, seed=5, stream_id=6, cols=True,
                                      rnd_t=1, stream_id_t=7)
    none, rows, amax, only = snip.gemm_requant(snip.NVFP4, a, b, M, N, K, g, seed=5, want_d=False, rows=False,
                                               cols=True, rnd_t=1, stream_id_t=7)
    torch.cuda.synchronize()
    assert none is None and rows is None
    np.testing.assert_array_equal(only.codes.cpu().numpy(), both.codes.cpu().numpy())
    np.testing.assert_array_equal(only.scales.cpu().numpy(), both.scales.cpu().numpy())
    # dW_prev = dY^T X: dY^T (N x M, blocks along M) times X^T quantized along M
    X = inputs.normal_bf16((M, 384), 1.0, 15, 3).cuda()
    xt = snip.quantize_nvfp4(X, orient=snip.ALONG_ROWS, rnd=1, seed=5, stream_id=8, layout=snip.MMA)
    D = snip.gemm(snip.NVFP4, a, b, M, N, K)
    torch.cuda.synchronize()
    lib = snip.quantize_nvfp4(D.to(torch.bfloat16), orient=snip.ALONG_ROWS, rnd=1, seed=5, stream_id=7, g_in=g,
                              layout=snip.MMA)
    out_fused = snip.gemm(snip.NVFP4, only, xt, N, 384, M)
    out_lib = snip.gemm(snip.NVFP4, lib, xt, N, 384, M)
    torch.cuda.synchronize()
    assert torch.equal(out_fused, out_lib)


# ---------------------------------------------------------------- exact products: bit-exact against the oracle

def _exact_operand(fmt, rows, K, seed):
    """A bf16 rows x K operand whose quantization is exact and whose GEMM
    products sum exactly in fp32 in any order.  NVFP4: every 16-block holds
    one +-6 and random E2M1 values, all times 448 * 2^-10, so the tensor scale
    g = amax / 2688 = 2^-10 and every block scale is 448: the MMA's partial
    sums are 448^2 times sums of E2M1 products (at most 22 bits).  FP8: E4M3
    values with exponents 6..8 (64 .. 448) and zeros, one 448, all times
    2^-8, so s = amax / 448 = 2^-8 and products are multiples of 64 below
    2^18 (sums of up to 512 of them stay below 2^24)."""
    rng = np.random.default_rng(seed)
    if fmt == 1:
        grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
        v = grid[rng.integers(0, 8, size=(rows, K))] * rng.choice([-1.0, 1.0], size=(rows, K))
        blk = v.reshape(rows, K // 16, 16)
        pos = rng.integers(0, 16, size=(rows, K // 16))
        np.put_along_axis(blk, pos[..., None], rng.choice([-6.0, 6.0], size=(rows, K // 16, 1)), axis=2)
        x = blk.reshape(rows, K) * 448.0 * 2.0 ** -10
    else:
        m = rng.integers(0, 8, size=(rows, K))
        e = rng.integers(6, 9, size=(rows, K))
        m = np.where(e == 8, np.minimum(m, 6), m)          # 1.75 * 2^8 = 448 is the largest
        v = (1 + m / 8.0) * 2.0 ** e * rng.choice([-1.0, 1.0], size=(rows, K))
        v = np.where(rng.random((rows, K)) < 0.2, 0.0, v)
        v[rng.integers(0, rows), rng.integers(0, K)] = 448.0
        x = v * 2.0 ** -8
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(t.float().numpy().astype(np.float64), x)   # exact in bf16
    return t


@pytest.mark.parametrize("fmt", [1, 0])
@pytest.mark.parametrize("M,N,K", [(192, 160, 256), (272, 400, 336), (2048, 2560, 512)])
@pytest.mark.parametrize("rnd,rnd_t", [(0, 0), (1, 1), (0, 1)])
def test_requant_bit_exact_vs_oracle_on_exact_products(snip, fmt, M, N, K, rnd, rnd_t):
    A = _exact_operand(fmt, M, K, 100 + M)
    B = _exact_operand(fmt, N, K, 200 + N)
    fname = "nvfp4" if fmt == 1 else "fp8"
    q = snip.quantize_nvfp4 if fmt == 1 else snip.quantize_fp8
    a = q(A.cuda(), rnd=1, seed=1, stream_id=2, layout=snip.MMA)
    b = q(B.cuda(), rnd=1, seed=1, stream_id=3, layout=snip.MMA)
    ref = oracle.gemm_tn(oracle.quantize(fname, A, 0, 1, 1, 2).dequant(), oracle.quantize(fname, B, 0, 1, 1, 3).dequant())
    assert np.array_equal(ref.astype(np.float32).astype(np.float64), ref)   # the product is exact in fp32
    gval = np.float32(0.8 * float(np.abs(ref).max()) / 2688.0)
    g = torch.tensor([gval], dtype=torch.float32, device="cuda")
    D, rq, amax, rq_t = snip.gemm_requant(fmt, a, b, M, N, K, g, rnd=rnd, seed=9, stream_id=21, cols=True,
                                          rnd_t=rnd_t, stream_id_t=23)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(D.cpu().numpy().astype(np.float64), ref)
    refb = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16)
    orc = oracle.quantize_nvfp4(refb, orient=0, rnd=rnd, seed=9, stream_id=21, g_in=float(gval))
    orc_t = oracle.quantize_nvfp4(refb, orient=1, rnd=rnd_t, seed=9, stream_id=23, g_in=float(gval))
    _, codes = mma_codes_to_rowmajor(rq.codes, M, N, fmt_nvfp4=True)
    _, scales = mma_scales_to_rowmajor(rq.scales, M, N)
    np.testing.assert_array_equal(codes, orc.codes)
    np.testing.assert_array_equal(scales, orc.scales)
    _, codes_t = mma_codes_to_rowmajor(rq_t.codes, N, M, fmt_nvfp4=True)
    _, scales_t = mma_scales_to_rowmajor(rq_t.scales, N, M)
    np.testing.assert_array_equal(codes_t, orc_t.codes)
    np.testing.assert_array_equal(scales_t, orc_t.scales)
    assert float(amax.cpu()) == float(refb.float().abs().max())


def test_requant_argument_errors(snip):
    import ctypes
    M, N, K = 200, 256, 256   # M not a multiple of 16: no column blocks
    a, b, _ = _operands(snip, 1, 208, N, K, 16)
    g = torch.tensor([1e-3], dtype=torch.float32, device="cuda")
    buf = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    ws = snip.small_workspace()
    L = snip.load()

    def call(rq, m=M):
        return L.snip_gemm_requant(snip.NVFP4, a.codes.data_ptr(), a.scales.data_ptr(), a.g.data_ptr(),
                                   b.codes.data_ptr(), b.scales.data_ptr(), b.g.data_ptr(), m, N, K, None, N,
                                   ctypes.byref(rq), ws.ptr, ws.nbytes, None)

    p = buf.data_ptr()
    assert call(snip.SnipRequant(g.data_ptr(), 0, 0, 0, None, None, None, 0, 0, p, p)) == snip.SNIP_ERR_SHAPE
    assert call(snip.SnipRequant(g.data_ptr(), 0, 0, 0, None, None, None, 0, 0, None, None)) == \
        snip.SNIP_ERR_INVALID_ARG
    assert call(snip.SnipRequant(g.data_ptr(), 0, 0, 0, None, None, None, 0, 0, p, None), 208) == \
        snip.SNIP_ERR_INVALID_ARG
    assert call(snip.SnipRequant(g.data_ptr(), 0, 0, 0, None, None, None, 2, 0, p, p), 208) == \
        snip.SNIP_ERR_INVALID_ARG
    torch.cuda.synchronize()
