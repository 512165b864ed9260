"""GPU parity of SNIP's statistics pass (error norms of NVFP4 and FP8
quantization, expected SR variance, per-block errors, the sqrt(3) check)
against the oracle, within 1e-4 relative."""
import math

import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import STATS_REL, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


def _check(snip, x, rnd, seed=0, sid=0, blocks=True, precomputed=False):
    xd = x.cuda()
    sc = snip.tensor_scales(xd) if precomputed else None
    raw, (b4, b8) = snip.quant_stats(xd, rnd=rnd, seed=seed, stream_id=sid, want_block_err=blocks, scales=sc)
    got = raw.cpu().numpy()
    ref = oracle.quant_stats(x, rnd=rnd, seed=seed, stream_id=sid, want_block_err=blocks)
    r = ref["raw"]
    for k in range(7):
        assert got[k] == pytest.approx(r[k], rel=STATS_REL, abs=1e-300), (k, got[k], r[k])
    if blocks:
        np.testing.assert_allclose(b4.cpu().numpy(), ref["block_err_nvfp4"], rtol=STATS_REL, atol=1e-30)
        np.testing.assert_allclose(b8.cpu().numpy(), ref["block_err_fp8"], rtol=STATS_REL, atol=1e-30)
    st = snip.snip_stats_finalize(got)
    assert (st.below_sqrt3_nvfp4 == 1) == ref["below_sqrt3_nvfp4"]
    if math.isfinite(ref["ratio_nvfp4"]):
        assert st.ratio_nvfp4 == pytest.approx(ref["ratio_nvfp4"], rel=STATS_REL)
    return got


@pytest.mark.parametrize("shape", [(64, 128), (272, 400), (1024, 2048)])
@pytest.mark.parametrize("rnd", [0, 1])
def test_stats_normal(snip, shape, rnd):
    _check(snip, inputs.normal_bf16(shape, 1e-3, 3, 7), rnd, seed=2, sid=18)
    _check(snip, inputs.normal_bf16(shape, 1.0, 3, 8), rnd, seed=2, sid=18, precomputed=True)


def test_stats_outliers(snip):
    _check(snip, inputs.outlier_bf16(512, 1024, seed=1, tensor_id=5, frac=0.001), 0)
    _check(snip, inputs.outlier_bf16(512, 1024, seed=1, tensor_id=5, frac=0.001), 1, seed=4, sid=3)


def test_stats_zero_and_grid(snip):
    z = _check(snip, torch.zeros((16, 64), dtype=torch.bfloat16), 0)
    assert z[0] == 0 and z[1] == 0 and z[2] == 0
    row = np.zeros(32, dtype=np.float32)
    row[0] = 2688.0
    row[16:20] = [6.0, -3.0, 1.5, 0.5]
    g = _check(snip, torch.tensor(row[None, :]).to(torch.bfloat16), 0)
    assert g[1] == 0.0 and g[3] == 0.0


def test_stats_nonfinite(snip):
    ws = snip.Workspace(snip.snip_quantize_workspace_size(0, 0))
    x = torch.ones((16, 32), dtype=torch.bfloat16)
    x[0, 0] = float("nan")
    raw, _ = snip.quant_stats(x.cuda(), ws=ws)
    assert ws.status() == snip.SNIP_ERR_NONFINITE
    assert np.all(np.isnan(raw.cpu().numpy()))


@pytest.mark.slow
def test_stats_outlier_sweep_full_size(snip):
    x = inputs.outlier_bf16(8192, 8192, seed=0, tensor_id=100)
    _check(snip, x, 0, blocks=False)
    _check(snip, x, 1, seed=1, sid=2, blocks=True)


@pytest.mark.parametrize("fmt", [1, 0])
@pytest.mark.parametrize("rnd", [0, 1])
@pytest.mark.parametrize("shape", [(272, 400), (1024, 2048)])
def test_fused_quantize_stats(snip, fmt, rnd, shape):
    """The fused pass writes the same codes as the plain quantizer and the same
    statistics as the oracle (blocks along cols, this call's rounding)."""
    x = inputs.outlier_bf16(shape[0], shape[1], seed=6, tensor_id=3, frac=0.002)
    xd = x.cuda()
    codes, scales, raw = snip.quantize_stats(fmt, xd, rnd=rnd, seed=7, stream_id=10)
    q = (snip.quantize_nvfp4 if fmt == 1 else snip.quantize_fp8)(xd, rnd=rnd, seed=7, stream_id=10,
                                                                   layout=snip.MMA)
    assert torch.equal(codes, q.codes)
    if fmt == 1:
        assert torch.equal(scales, q.scales)
    ref = oracle.quant_stats(x, rnd=rnd, seed=7, stream_id=10)["raw"]
    got = raw.cpu().numpy()
    for k in range(7):
        assert got[k] == pytest.approx(ref[k], rel=STATS_REL, abs=1e-300), (k, got[k], ref[k])


def test_qlinear_stats_outputs(snip):
    """snip_qlinear_fwd/bwd statistics outputs equal SNIP's statistics of X, W
    (forward rounding) and dY (dgrad rounding, stream layer*8+2)."""
    X, W, dY = inputs.single_linear_inputs(272, 400, 336, seed=8)
    layer, seed = 1, 4
    for code in (1, 0):
        plan = snip.Plan([code, code], seed=seed)
        ws = snip.qlinear_workspace(plan, layer, 272, 400, 336)
        sf = torch.empty((2, snip.STATS_NVALS), dtype=torch.float64, device="cuda")
        sb = torch.empty(snip.STATS_NVALS, dtype=torch.float64, device="cuda")
        snip.qlinear_fwd(plan, layer, X.cuda(), W.cuda(), ws, stats=sf)
        snip.qlinear_bwd(plan, layer, X.cuda(), W.cuda(), dY.cuda(), ws, stats=sb)
        torch.cuda.synchronize()
        assert ws.status() == snip.SNIP_OK
        refs = [oracle.quant_stats(X)["raw"], oracle.quant_stats(W)["raw"],
                oracle.quant_stats(dY, rnd=1, seed=seed, stream_id=layer * 8 + 2)["raw"]]
        for got, ref in zip([sf[0].cpu().numpy(), sf[1].cpu().numpy(), sb.cpu().numpy()], refs):
            for k in range(7):
                assert got[k] == pytest.approx(ref[k], rel=STATS_REL, abs=1e-300), (k, got[k], ref[k])
