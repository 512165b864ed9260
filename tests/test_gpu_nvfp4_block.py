"""GPU parity of NVFP4 with longer blocks (32, 64, 128 E2M1 values per E4M3
scale; the block-size axis of the FP4 study in "FP4 all the way", Outline)
against the oracle: codes bit-exact and each block's scale repeated over its
16-element sub-blocks, in both layouts, orientations and roundings; the
operands through the NVFP4 GEMM and the quantized linear layer under a
longer-block plan within the GEMM tolerance; block 16 equals NVFP4; shape and
argument errors."""
import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import STATS_REL, gemm_close, mma_codes_to_rowmajor, mma_scales_to_rowmajor, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


def _x(shape, seed):
    # rows with sub-blocks of very different magnitudes, so block maxima come from different sub-blocks
    x = inputs.normal_bf16(shape, 1.0, seed, 1).float()
    g = torch.Generator().manual_seed(seed)
    x = x * torch.exp2(torch.randint(-6, 7, (shape[0], shape[1] // 16), generator=g).float()).repeat_interleave(16, 1)
    x[-1, :16] = 0.0
    return x.to(torch.bfloat16)


def _expand(scales, block):
    return np.repeat(scales, block // 16, axis=1)


@pytest.mark.parametrize("block", [32, 64, 128])
@pytest.mark.parametrize("shape", [(128, 256), (384, 640), (1024, 1536)])
@pytest.mark.parametrize("orient", [0, 1])
@pytest.mark.parametrize("rnd", [0, 1])
def test_block_rowmajor_bit_exact(snip, block, shape, orient, rnd):
    x = _x(shape, shape[0] + block)
    q = snip.quantize_nvfp4_block(x.cuda(), block, orient=orient, rnd=rnd, seed=4, stream_id=9)
    torch.cuda.synchronize()
    ref = oracle.quantize_nvfp4_block(x, block, orient=orient, rnd=rnd, seed=4, stream_id=9)
    np.testing.assert_array_equal(q.codes.cpu().numpy().reshape(ref.codes.shape), ref.codes)
    np.testing.assert_array_equal(q.scales.cpu().numpy().reshape(ref.rows, -1), _expand(ref.scales, block))
    assert float(q.g.cpu()) == ref.g


@pytest.mark.parametrize("block", [32, 128])
@pytest.mark.parametrize("shape", [(384, 640), (256, 1280)])
@pytest.mark.parametrize("orient", [0, 1])
@pytest.mark.parametrize("rnd", [0, 1])
def test_block_mma_layout_bit_exact(snip, block, shape, orient, rnd):
    x = _x(shape, 7 * shape[0] + block)
    q = snip.quantize_nvfp4_block(x.cuda(), block, orient=orient, rnd=rnd, seed=1, stream_id=3, layout=snip.MMA)
    torch.cuda.synchronize()
    ref = oracle.quantize_nvfp4_block(x, block, orient=orient, rnd=rnd, seed=1, stream_id=3)
    full, real = mma_codes_to_rowmajor(q.codes, q.out_rows, q.out_cols, fmt_nvfp4=True)
    np.testing.assert_array_equal(real, ref.codes)
    np.testing.assert_array_equal(full[q.out_rows:], 0)
    np.testing.assert_array_equal(full[:, q.out_cols // 2:], 0)
    sfull, sreal = mma_scales_to_rowmajor(q.scales, q.out_rows, q.out_cols)
    np.testing.assert_array_equal(sreal, _expand(ref.scales, block))


def test_block16_is_nvfp4(snip):
    x = _x((256, 512), 3).cuda()
    for orient in (0, 1):
        a = snip.quantize_nvfp4(x, orient=orient, rnd=1, seed=2, stream_id=5, layout=snip.MMA)
        b = snip.quantize_nvfp4_block(x, 16, orient=orient, rnd=1, seed=2, stream_id=5, layout=snip.MMA)
        torch.cuda.synchronize()
        assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)


@pytest.mark.parametrize("block", [32, 64])
@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (2048, 2560, 512)])
def test_block_gemm(snip, block, M, N, K):
    """Longer-block operands through the NVFP4 GEMM (one-CTA and CTA-pair kernels)."""
    X = inputs.normal_bf16((M, K), 1.0, 21, 1)
    W = inputs.normal_bf16((N, K), 0.02, 21, 2)
    a = snip.quantize_nvfp4_block(X.cuda(), block, layout=snip.MMA)
    b = snip.quantize_nvfp4_block(W.cuda(), block, layout=snip.MMA)
    fmt = {32: snip.NVFP4_B32, 64: snip.NVFP4_B64}[block]
    D = snip.gemm(fmt, a, b, M, N, K).cpu().numpy()
    ref = oracle.gemm_tn(oracle.quantize_nvfp4_block(X, block).dequant(), oracle.quantize_nvfp4_block(W, block).dequant())
    gemm_close(D, ref, f"nvfp4-b{block} {M}x{N}x{K}")


@pytest.mark.parametrize("fmt,name", [(5, "nvfp4-b32"), (6, "nvfp4-b64"), (7, "nvfp4-b128")])
def test_block_qlinear(snip, fmt, name):
    T, K, N = 256, 384, 512
    X, W, dY = inputs.single_linear_inputs(T, K, N, seed=8)
    layer, seed = 1, 3
    plan = snip.Plan([snip.NVFP4, fmt], seed=seed)
    ws = snip.qlinear_workspace(plan, layer, T, K, N)
    Xd, Wd, dYd = X.cuda(), W.cuda(), dY.cuda()
    sf = torch.empty((2, snip.STATS_NVALS), dtype=torch.float64, device="cuda")
    sb = torch.empty(snip.STATS_NVALS, dtype=torch.float64, device="cuda")
    Y = snip.qlinear_fwd(plan, layer, Xd, Wd, ws, stats=sf)
    dX, dW = snip.qlinear_bwd(plan, layer, Xd, Wd, dYd, ws, stats=sb)
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK
    gemm_close(Y.cpu().numpy(), oracle.qlinear_fwd(name, X, W, layer=layer, seed=seed), "Y")
    gemm_close(dX.cpu().numpy(), oracle.qlinear_dgrad(name, dY, W, layer=layer, seed=seed), "dX")
    gemm_close(dW.cpu().numpy(), oracle.qlinear_wgrad(name, dY, X, layer=layer, seed=seed), "dW")
    # SNIP's statistics (NVFP4 and FP8 candidates) of the layer's tensors, as for any format
    refs = [oracle.quant_stats(X)["raw"], oracle.quant_stats(W)["raw"],
            oracle.quant_stats(dY, rnd=1, seed=seed, stream_id=layer * 8 + 2)["raw"]]
    for got, ref in zip([sf[0].cpu().numpy(), sf[1].cpu().numpy(), sb.cpu().numpy()], refs):
        for k in range(7):
            assert got[k] == pytest.approx(ref[k], rel=STATS_REL, abs=1e-300), (k, got[k], ref[k])


def test_block_errors(snip):
    x = torch.zeros((64, 96), dtype=torch.bfloat16, device="cuda")   # 96 is not a multiple of 64
    with pytest.raises(snip.SnipError) as e:
        snip.quantize_nvfp4_block(x, 64)
    assert e.value.status == snip.SNIP_ERR_SHAPE
    with pytest.raises(snip.SnipError) as e:
        snip.quantize_nvfp4_block(x, 48)
    assert e.value.status == snip.SNIP_ERR_INVALID_ARG
    plan = snip.Plan([snip.NVFP4_B128], seed=0)
    with pytest.raises(snip.SnipError) as e:   # K = 64 is not a multiple of 128
        snip.qlinear_fwd(plan, 0, torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda"),
                         torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda"), snip.Workspace(1 << 22))
    assert e.value.status == snip.SNIP_ERR_SHAPE


@pytest.mark.parametrize("fmt,block", [(5, 32), (7, 128)])
@pytest.mark.parametrize("rnd", [0, 1])
def test_block_quantize_stats_fused(snip, fmt, block, rnd):
    """Longer-block codes and SNIP's statistics of the candidate formats from one pass."""
    x = _x((256, 1024), 40 + block)
    codes, scales, raw = snip.quantize_stats(fmt, x.cuda(), rnd=rnd, seed=6, stream_id=13, layout=snip.ROWMAJOR)
    torch.cuda.synchronize()
    ref = oracle.quantize_nvfp4_block(x, block, rnd=rnd, seed=6, stream_id=13)
    np.testing.assert_array_equal(codes.cpu().numpy().reshape(ref.codes.shape), ref.codes)
    np.testing.assert_array_equal(scales.cpu().numpy().reshape(ref.rows, -1), _expand(ref.scales, block))
    r = oracle.quant_stats(x, rnd=rnd, seed=6, stream_id=13)["raw"]
    got = raw.cpu().numpy()
    for k in range(7):
        assert got[k] == pytest.approx(r[k], rel=STATS_REL, abs=1e-300), k
