"""GPU parity of the FP8 E5M2 gradient variant against the oracle: E5M2 codes
and tensor scale bit-exact in both layouts, orientations and roundings; the
mixed E5M2 x E4M3 GEMM on both kernels; the quantized linear layer under a
plan whose layer format keeps E4M3 forward and quantizes dY, dY^T in E5M2."""
import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import STATS_REL, gemm_close, mma_codes_to_rowmajor, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


def _g(shape, seed, sigma):
    x = inputs.normal_bf16(shape, sigma, seed, 3).float()
    x[0, :16] = 0.0
    x[1, 3] = -0.0
    x[2, :8] *= 1e4                       # wide range: the tensor max sits far above most values
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("shape", [(32, 48), (144, 272), (512, 1024)])
@pytest.mark.parametrize("orient", [0, 1])
@pytest.mark.parametrize("rnd", [0, 1])
@pytest.mark.parametrize("layout", [0, 1])
def test_e5m2_bit_exact(snip, shape, orient, rnd, layout):
    x = _g(shape, sum(shape), 1e-3)
    q = snip.quantize_e5m2(x.cuda(), orient=orient, rnd=rnd, seed=4, stream_id=9, layout=layout)
    torch.cuda.synchronize()
    ref = oracle.quantize_e5m2(x, orient=orient, rnd=rnd, seed=4, stream_id=9)
    assert float(q.s.cpu()) == ref.s
    if layout == 0:
        np.testing.assert_array_equal(q.codes.cpu().numpy().reshape(ref.codes.shape), ref.codes)
    else:
        full, real = mma_codes_to_rowmajor(q.codes, q.out_rows, q.out_cols, fmt_nvfp4=False)
        np.testing.assert_array_equal(real, ref.codes)
        np.testing.assert_array_equal(full[q.out_rows:], 0)


def test_e5m2_with_given_amax(snip):
    x = _g((64, 64), 5, 1.0)
    sc = snip.tensor_scales(x.cuda())
    q = snip.quantize_e5m2(x.cuda(), amax_in=sc[0:1], rnd=1, seed=2, stream_id=1)
    ref = oracle.quantize_e5m2(x, rnd=1, seed=2, stream_id=1)
    np.testing.assert_array_equal(q.codes.cpu().numpy().reshape(ref.codes.shape), ref.codes)


@pytest.mark.parametrize("M,N,K", [(200, 176, 320), (2048, 2560, 512)])
def test_e5m2_e4m3_gemm(snip, M, N, K):
    dY = _g((M, K), 7, 1e-3)
    W = inputs.normal_bf16((N, K), 0.02, 7, 2)
    a = snip.quantize_e5m2(dY.cuda(), rnd=1, seed=1, stream_id=2, layout=snip.MMA)
    b = snip.quantize_fp8(W.cuda(), layout=snip.MMA)
    D = snip.gemm(snip.FP8_E5M2, a, b, M, N, K).cpu().numpy()
    ref = oracle.gemm_tn(oracle.quantize_e5m2(dY, rnd=1, seed=1, stream_id=2).dequant(), oracle.quantize_fp8(W).dequant())
    gemm_close(D, ref, f"e5m2 x e4m3 {M}x{N}x{K}")


@pytest.mark.parametrize("shape", [(64, 128, 128), (272, 400, 336), (1024, 2048, 768)])
def test_qlinear_e5m2_gradients(snip, shape):
    T, K, N = shape
    X, W, dY = inputs.single_linear_inputs(T, K, N, seed=5)
    layer, seed = 1, 8
    plan = snip.Plan([snip.FP8, snip.FP8_E5M2_GRAD], seed=seed)
    ws = snip.qlinear_workspace(plan, layer, T, K, N)
    Xd, Wd, dYd = X.cuda(), W.cuda(), dY.cuda()
    sf = torch.empty((2, snip.STATS_NVALS), dtype=torch.float64, device="cuda")
    sb = torch.empty(snip.STATS_NVALS, dtype=torch.float64, device="cuda")
    Y = snip.qlinear_fwd(plan, layer, Xd, Wd, ws, stats=sf)
    dX, dW = snip.qlinear_bwd(plan, layer, Xd, Wd, dYd, ws, stats=sb)
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK
    sid = lambda tag: oracle.stream_id(layer, tag)
    gemm_close(Y.cpu().numpy(), oracle.qlinear_fwd("fp8", X, W, layer=layer, seed=seed), "Y")
    dyq = oracle.quantize_e5m2(dY, 0, oracle.SR, seed, sid(2)).dequant()
    wtq = oracle.quantize_fp8(W, 1, oracle.SR, seed, sid(3)).dequant()
    gemm_close(dX.cpu().numpy(), oracle.gemm_tn(dyq, wtq), "dX")
    dytq = oracle.quantize_e5m2(dY, 1, oracle.SR, seed, sid(4)).dequant()
    xtq = oracle.quantize_fp8(X, 1, oracle.SR, seed, sid(5)).dequant()
    gemm_close(dW.cpu().numpy(), oracle.gemm_tn(dytq, xtq), "dW")
    refs = [oracle.quant_stats(X)["raw"], oracle.quant_stats(W)["raw"],
            oracle.quant_stats(dY, rnd=1, seed=seed, stream_id=sid(2))["raw"]]
    for got, ref in zip([sf[0].cpu().numpy(), sf[1].cpu().numpy(), sb.cpu().numpy()], refs):
        for k in range(7):
            assert got[k] == pytest.approx(ref[k], rel=STATS_REL, abs=1e-300), (k, got[k], ref[k])


def test_plan_rejects_operand_format(snip):
    with pytest.raises(snip.SnipError):
        snip.Plan([snip.FP8_E5M2], seed=0)


@pytest.mark.parametrize("rnd", [0, 1])
def test_e5m2_quantize_stats_fused(snip, rnd):
    """E5M2 codes and SNIP's statistics of the candidate formats (NVFP4, E4M3) from one pass."""
    x = inputs.normal_bf16((256, 768), 1e-3, 17, 1)
    codes, _, raw = snip.quantize_stats(snip.FP8_E5M2, x.cuda(), rnd=rnd, seed=4, stream_id=10,
                                        layout=snip.ROWMAJOR)
    torch.cuda.synchronize()
    ref = oracle.quantize_e5m2(x, rnd=rnd, seed=4, stream_id=10)
    np.testing.assert_array_equal(codes.cpu().numpy().reshape(ref.codes.shape), ref.codes)
    r = oracle.quant_stats(x, rnd=rnd, seed=4, stream_id=10)["raw"]
    got = raw.cpu().numpy()
    for k in range(7):
        assert got[k] == pytest.approx(r[k], rel=STATS_REL, abs=1e-300), k
