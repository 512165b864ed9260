"""GPU parity of the MXFP4 variant (OCP Microscaling v1.0: 32 E2M1 values per
E8M0 power-of-two scale, no tensor scale) against the oracle: codes and
scales bit-exact in both layouts, orientations and roundings; the
block-scaled GEMM (scale_vec::2X, UE8M0) on both kernels within the GEMM
tolerance; the quantized linear layer under an MXFP4 plan; statistics next
to MXFP4 codes; shape and non-finite errors."""
import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import STATS_REL, gemm_close, mma_codes_to_rowmajor, mma_mx_scales_to_rowmajor, need_gpu

pytestmark = pytest.mark.gpu

SHAPES = [(32, 64), (96, 160), (256, 512), (288, 480), (1024, 2048)]


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


def _x(shape, seed, sigma=1.0):
    x = inputs.normal_bf16(shape, sigma, seed, 1)
    g = torch.Generator().manual_seed(seed)
    # a few blocks spanning many binades (block scales from 2^-127 up), zeros and negative zeros
    x = x.float()
    x[: shape[0] // 4] *= torch.exp2(torch.randint(-40, 40, (shape[0] // 4, 1), generator=g).float())
    x[-1, :32] = 0.0
    x[-1, 32:64] = -0.0
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("orient", [0, 1])
@pytest.mark.parametrize("rnd", [0, 1])
def test_mxfp4_rowmajor_bit_exact(snip, shape, orient, rnd):
    rows, cols = shape
    x = _x(shape, rows + cols)
    q = snip.quantize_mxfp4(x.cuda(), orient=orient, rnd=rnd, seed=9, stream_id=5)
    torch.cuda.synchronize()
    ref = oracle.quantize_mxfp4(x, orient=orient, rnd=rnd, seed=9, stream_id=5)
    np.testing.assert_array_equal(q.codes.cpu().numpy().reshape(ref.codes.shape), ref.codes)
    np.testing.assert_array_equal(q.scales.cpu().numpy().reshape(ref.scales.shape), ref.scales)


@pytest.mark.parametrize("shape", [(96, 160), (288, 480), (512, 768)])
@pytest.mark.parametrize("orient", [0, 1])
@pytest.mark.parametrize("rnd", [0, 1])
def test_mxfp4_mma_layout_bit_exact(snip, shape, orient, rnd):
    rows, cols = shape
    x = _x(shape, 3 * rows + cols)
    q = snip.quantize_mxfp4(x.cuda(), orient=orient, rnd=rnd, seed=2, stream_id=7, layout=snip.MMA)
    torch.cuda.synchronize()
    ref = oracle.quantize_mxfp4(x, orient=orient, rnd=rnd, seed=2, stream_id=7)
    full, real = mma_codes_to_rowmajor(q.codes, q.out_rows, q.out_cols, fmt_nvfp4=True)
    np.testing.assert_array_equal(real, ref.codes)
    np.testing.assert_array_equal(full[q.out_rows:], 0)             # padding rows encode zeros
    np.testing.assert_array_equal(full[:, q.out_cols // 2:], 0)      # padding contraction encodes zeros
    sfull, sreal = mma_mx_scales_to_rowmajor(q.scales, q.out_rows, q.out_cols)
    np.testing.assert_array_equal(sreal, ref.scales)


@pytest.mark.parametrize("M,N,K", [(200, 176, 320), (64, 128, 128), (2048, 2560, 512), (2000, 2512, 288)])
def test_mxfp4_gemm(snip, M, N, K):
    """Both GEMM kernels: the small shapes run on the one-CTA kernel, the
    large ones on the CTA pair (a wave of 256 x 256 tiles)."""
    X = inputs.normal_bf16((M, K), 1.0, 11, 1)
    W = inputs.normal_bf16((N, K), 0.02, 11, 2)
    a = snip.quantize_mxfp4(X.cuda(), layout=snip.MMA)
    b = snip.quantize_mxfp4(W.cuda(), layout=snip.MMA)
    D = snip.gemm(snip.MXFP4, a, b, M, N, K).cpu().numpy()
    ref = oracle.gemm_tn(oracle.quantize_mxfp4(X).dequant(), oracle.quantize_mxfp4(W).dequant())
    gemm_close(D, ref, f"mxfp4 {M}x{N}x{K}")


def test_mxfp4_gemm_identity(snip):
    """A scaled identity B passes x-hat through: each MMA's two E8M0 scales
    (scale-factor IDs 0 and 2 of a chunk word) multiply the right blocks."""
    X = _x((192, 256), 21)
    I = torch.eye(256, dtype=torch.float32).mul(0.25).to(torch.bfloat16)
    a = snip.quantize_mxfp4(X.cuda(), layout=snip.MMA)
    b = snip.quantize_mxfp4(I.cuda(), layout=snip.MMA)
    D = snip.gemm(snip.MXFP4, a, b, 192, 256, 256).cpu().numpy()
    np.testing.assert_array_equal(D, oracle.quantize_mxfp4(X).dequant() * 0.25)


@pytest.mark.parametrize("shape", [(64, 128, 128), (288, 416, 352), (1024, 2048, 768)])
def test_mxfp4_qlinear(snip, shape):
    T, K, N = shape
    X, W, dY = inputs.single_linear_inputs(T, K, N, seed=4)
    layer, seed = 1, 6
    plan = snip.Plan([snip.MXFP4, snip.MXFP4], seed=seed)
    ws = snip.qlinear_workspace(plan, layer, T, K, N)
    Xd, Wd, dYd = X.cuda(), W.cuda(), dY.cuda()
    sf = torch.empty((2, snip.STATS_NVALS), dtype=torch.float64, device="cuda")
    sb = torch.empty(snip.STATS_NVALS, dtype=torch.float64, device="cuda")
    Y = snip.qlinear_fwd(plan, layer, Xd, Wd, ws, stats=sf)
    dX, dW = snip.qlinear_bwd(plan, layer, Xd, Wd, dYd, ws, stats=sb)
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK
    gemm_close(Y.cpu().numpy(), oracle.qlinear_fwd("mxfp4", X, W, layer=layer, seed=seed), "Y")
    gemm_close(dX.cpu().numpy(), oracle.qlinear_dgrad("mxfp4", dY, W, layer=layer, seed=seed), "dX")
    gemm_close(dW.cpu().numpy(), oracle.qlinear_wgrad("mxfp4", dY, X, layer=layer, seed=seed), "dW")
    # statistics of the layer's tensors come out as for the other formats
    refs = [oracle.quant_stats(X)["raw"], oracle.quant_stats(W)["raw"],
            oracle.quant_stats(dY, rnd=1, seed=seed, stream_id=layer * 8 + 2)["raw"]]
    for got, ref in zip([sf[0].cpu().numpy(), sf[1].cpu().numpy(), sb.cpu().numpy()], refs):
        for k in range(7):
            assert got[k] == pytest.approx(ref[k], rel=STATS_REL, abs=1e-300), (k, got[k], ref[k])


def test_mxfp4_quantize_stats(snip):
    x = _x((256, 512), 31)
    codes, scales, raw = snip.quantize_stats(snip.MXFP4, x.cuda(), rnd=1, seed=3, stream_id=12,
                                             layout=snip.ROWMAJOR)
    torch.cuda.synchronize()
    ref = oracle.quantize_mxfp4(x, rnd=1, seed=3, stream_id=12)
    np.testing.assert_array_equal(codes.cpu().numpy().reshape(ref.codes.shape), ref.codes)
    np.testing.assert_array_equal(scales.cpu().numpy().reshape(ref.scales.shape), ref.scales)
    r = oracle.quant_stats(x, rnd=1, seed=3, stream_id=12)["raw"]
    got = raw.cpu().numpy()
    for k in range(7):
        assert got[k] == pytest.approx(r[k], rel=STATS_REL, abs=1e-300), k


def test_mxfp4_errors(snip):
    x = torch.zeros((64, 48), dtype=torch.bfloat16, device="cuda")   # 48 is not a multiple of 32
    with pytest.raises(snip.SnipError) as e:
        snip.quantize_mxfp4(x)
    assert e.value.status == snip.SNIP_ERR_SHAPE
    with pytest.raises(snip.SnipError):
        snip.quantize_mxfp4(torch.zeros((48, 64), dtype=torch.bfloat16, device="cuda"), orient=1)
    plan = snip.Plan([snip.MXFP4], seed=0)
    with pytest.raises(snip.SnipError) as e:   # T = 48 is not a multiple of 32
        snip.qlinear_fwd(plan, 0, torch.zeros((48, 64), dtype=torch.bfloat16, device="cuda"),
                         torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda"), snip.Workspace(1 << 22))
    assert e.value.status == snip.SNIP_ERR_SHAPE
    xn = torch.ones((64, 64), dtype=torch.bfloat16)
    xn[3, 5] = float("nan")
    ws = snip.Workspace(snip.snip_quantize_workspace_size(0, 0))
    snip.quantize_mxfp4(xn.cuda(), ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_ERR_NONFINITE
