"""The weight-gradient form of the sqrt(3) check ("FP4 all the way",
Outline): the oracle's sums against closed forms (CPU), the host finalize,
and on the GPU the library's bf16 tensor-core GEMM with the two sums in its
epilogue against the oracle for NVFP4 and FP8 layers: tiles cut by N < 128
and K < 256, tokens not a multiple of the 64-token stage, several tiles per
CTA, and the 7B Down linear at full size."""
import math

import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs, snip as snip_mod


def test_oracle_closed_forms():
    X, _, dY = inputs.single_linear_inputs(64, 96, 80, seed=2)
    dw = dY.double().numpy().T @ X.double().numpy()
    ref, err = oracle.dw_noise(X, dY, dw)
    assert err == 0.0 and ref == pytest.approx(float(np.sum(dw * dw)), rel=1e-15)
    ref2, err2 = oracle.dw_noise(X, dY, dw * 1.25)          # error = 0.25 dW
    assert ref2 == ref and err2 == pytest.approx(0.0625 * ref, rel=1e-12)
    # bf16 widening is exact
    np.testing.assert_array_equal(oracle._bits_to_f64(X), X.double().numpy())


def test_finalize_host():
    assert snip_mod.snip_dw_noise_finalize([4.0, 1.0]) == (2.0, False)
    r, below = snip_mod.snip_dw_noise_finalize([2.0, 1.0])
    assert r == pytest.approx(math.sqrt(2.0)) and below
    assert snip_mod.snip_dw_noise_finalize([1.0, 0.0]) == (math.inf, False)
    with pytest.raises(snip_mod.SnipError):
        snip_mod.snip_dw_noise_finalize([float("nan"), 1.0])


@pytest.mark.gpu
@pytest.mark.parametrize("code,fmt", [(1, "nvfp4"), (0, "fp8")])
@pytest.mark.parametrize("shape", [(256, 128, 96), (1024, 512, 768), (272, 400, 336), (4096, 2048, 1280)])
def test_dw_noise_gpu(code, fmt, shape):
    from gpu_helpers import need_gpu
    snip = need_gpu()
    T, K, N = shape
    X, W, dY = inputs.single_linear_inputs(T, K, N, seed=7)
    layer, seed = 0, 3
    plan = snip.Plan([code], seed=seed)
    ws = snip.qlinear_workspace(plan, layer, T, K, N)
    Xd, dYd = X.cuda(), dY.cuda()
    _, dW = snip.qlinear_bwd(plan, layer, Xd, W.cuda(), dYd, ws)
    out = snip.dw_noise(Xd, dYd, dW).cpu().numpy()
    torch.cuda.synchronize()
    dwq_ref = oracle.qlinear_wgrad(fmt, dY, X, layer=layer, seed=seed)
    ref, err = oracle.dw_noise(X, dY, dwq_ref)
    assert out[0] == pytest.approx(ref, rel=1e-5)
    # the two quantized dW differ by at most the GEMM bound (1e-5 relative Frobenius), the two
    # full-precision dW by fp32 rounding: bound the error norms' difference by both
    bound = 2e-5 * (math.sqrt(float(np.sum(dwq_ref ** 2))) + math.sqrt(ref))
    assert abs(math.sqrt(out[1]) - math.sqrt(err)) <= bound
    # an exact dW (the oracle's, rounded to fp32) leaves only rounding error
    exact = torch.tensor(dY.double().numpy().T @ X.double().numpy(), dtype=torch.float32).cuda()
    out2 = snip.dw_noise(Xd, dYd, exact).cpu().numpy()
    assert out2[1] <= 1e-10 * out2[0]
    ratio, below = snip.snip_dw_noise_finalize(out)
    assert ratio == pytest.approx(math.sqrt(ref / err), rel=1e-3) and below == (ratio < math.sqrt(3))


@pytest.mark.gpu
@pytest.mark.slow
def test_dw_noise_llama7b_down_full():
    """T = 8192, K = 11008, N = 4096 (the 7B block's Down linear, NVFP4)."""
    from gpu_helpers import need_gpu
    snip = need_gpu()
    cfg = inputs.LLAMA7B
    j = [l.name for l in cfg.linears].index("Down")
    X, W, dY = inputs.linear_inputs(cfg, j, seed=0, device="cuda")
    T, K, N = cfg.T, cfg.linears[j].K, cfg.linears[j].N
    plan = snip.Plan([1] * len(cfg.linears), seed=0)
    ws = snip.qlinear_workspace(plan, j, T, K, N)
    _, dW = snip.qlinear_bwd(plan, j, X, W, dY, ws)
    out = snip.dw_noise(X, dY, dW).cpu().numpy()
    torch.cuda.synchronize()
    ref, err = oracle.dw_noise(X.cpu(), dY.cpu(), dW.cpu().numpy())
    # statistics bound (1e-4 relative); fp32 accumulation over 8192 tokens moves ||dW||^2 by ~2e-5
    from gpu_helpers import STATS_REL
    assert out[0] == pytest.approx(ref, rel=STATS_REL)
    assert out[1] == pytest.approx(err, rel=STATS_REL)
