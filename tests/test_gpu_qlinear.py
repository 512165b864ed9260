"""GPU parity of the three GEMMs of the quantized linear layer (SNIP Figure 5)
against the oracle's fp64 product of the same dequantized operands:
relative Frobenius error <= 1e-5 and max |diff| <= 1e-3 * rms, for NVFP4 and
FP8 layers, at the single-layer size, at ragged multi-tile sizes, through the
standalone GEMM entry point, and on sampled rows of the Llama-shaped blocks."""
import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import gemm_close, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


FMTS = [("nvfp4", 1), ("fp8", 0)]


def _run_layer(snip, fmt_code, X, W, dY, layer=0, seed=0):
    plan = snip.Plan([fmt_code] * (layer + 1), seed=seed)
    T, K = X.shape
    N = W.shape[0]
    ws = snip.qlinear_workspace(plan, layer, T, K, N)
    Xd, Wd, dYd = X.cuda(), W.cuda(), dY.cuda()
    Y = snip.qlinear_fwd(plan, layer, Xd, Wd, ws)
    dX, dW = snip.qlinear_bwd(plan, layer, Xd, Wd, dYd, ws)
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK
    return Y.cpu().numpy(), dX.cpu().numpy(), dW.cpu().numpy()


@pytest.mark.parametrize("fmt,code", FMTS)
@pytest.mark.parametrize("shape", [(64, 128, 128), (272, 400, 336), (1024, 2048, 768), (128, 256, 512)])
def test_qlinear_fwd_bwd(snip, fmt, code, shape):
    T, K, N = shape
    X, W, dY = inputs.single_linear_inputs(T, K, N, seed=1)
    layer = 2
    Y, dX, dW = _run_layer(snip, code, X, W, dY, layer=layer, seed=5)
    gemm_close(Y, oracle.qlinear_fwd(fmt, X, W, layer=layer, seed=5), f"{fmt} Y {shape}")
    gemm_close(dX, oracle.qlinear_dgrad(fmt, dY, W, layer=layer, seed=5), f"{fmt} dX {shape}")
    gemm_close(dW, oracle.qlinear_wgrad(fmt, dY, X, layer=layer, seed=5), f"{fmt} dW {shape}")


@pytest.mark.parametrize("fmt,code", FMTS)
def test_standalone_gemm_identity_and_random(snip, fmt, code):
    """snip_gemm on quantizer outputs: a scaled identity passes x-hat through,
    and a random pair matches the fp64 product."""
    X = inputs.normal_bf16((200, 320), 1.0, 3, 1)
    W = torch.eye(320, dtype=torch.float32).mul(0.5).to(torch.bfloat16)
    q = snip.quantize_nvfp4 if code == 1 else snip.quantize_fp8
    a = q(X.cuda(), layout=snip.MMA)
    b = q(W.cuda(), layout=snip.MMA)
    D = snip.gemm(code, a, b, 200, 320, 320).cpu().numpy()
    ref = oracle.gemm_tn(oracle.quantize(fmt, X).dequant(), oracle.quantize(fmt, W).dequant())
    gemm_close(D, ref, f"{fmt} identity")
    B = inputs.normal_bf16((176, 320), 0.02, 3, 2)
    bb = q(B.cuda(), layout=snip.MMA)
    D2 = snip.gemm(code, a, bb, 200, 176, 320).cpu().numpy()
    gemm_close(D2, oracle.gemm_tn(oracle.quantize(fmt, X).dequant(), oracle.quantize(fmt, B).dequant()),
               f"{fmt} random")


@pytest.mark.parametrize("fmt,code", FMTS)
@pytest.mark.parametrize("shape", [(2048, 2560, 512), (2000, 2512, 272)])
def test_gemm_cta_pair_path(snip, fmt, code, shape):
    """GEMMs with at least one 256 x 256 tile per SM pair run on the CTA-pair
    kernel: an exact wave of tiles and a ragged one (M, N not multiples of
    256, K not a multiple of the 256-element stage)."""
    M, N, K = shape
    assert ((M + 255) // 256) * ((N + 255) // 256) >= torch.cuda.get_device_properties(0).multi_processor_count // 2
    X = inputs.normal_bf16((M, K), 1.0, 6, 1)
    W = inputs.normal_bf16((N, K), 0.02, 6, 2)
    q = snip.quantize_nvfp4 if code == 1 else snip.quantize_fp8
    D = snip.gemm(code, q(X.cuda(), layout=snip.MMA), q(W.cuda(), layout=snip.MMA), M, N, K).cpu().numpy()
    gemm_close(D, oracle.gemm_tn(oracle.quantize(fmt, X).dequant(), oracle.quantize(fmt, W).dequant()),
               f"{fmt} pair {shape}")


@pytest.mark.parametrize("shape,e5m2", [((4864, 2048, 16384), False), ((4800, 2000, 16400), True)])
def test_gemm_fp8_wide_pair_tiles(snip, shape, e5m2):
    """FP8 GEMMs with long contractions whose 256 x 512 pair tiles fill whole waves of SM pairs
    run two N = 256 MMAs per k-step (19 x 4 tiles on 76 pairs): an exact case and a ragged one
    (M, N not multiples of the tile, N's last 512-column tile partly past N, K not a multiple of
    the 128-element stage); A in E4M3 or E5M2."""
    M, N, K = shape
    X = inputs.normal_bf16((M, K), 1.0, 9, 1)
    W = inputs.normal_bf16((N, K), 0.02, 9, 2)
    if e5m2:
        a = snip.quantize_e5m2(X.cuda(), layout=snip.MMA)
        ref_a = oracle.quantize_e5m2(X)
    else:
        a = snip.quantize_fp8(X.cuda(), layout=snip.MMA)
        ref_a = oracle.quantize_fp8(X)
    b = snip.quantize_fp8(W.cuda(), layout=snip.MMA)
    D = snip.gemm(snip.FP8_E5M2 if e5m2 else snip.FP8, a, b, M, N, K).cpu().numpy()
    gemm_close(D, oracle.gemm_tn(ref_a.dequant(), oracle.quantize_fp8(W).dequant()), f"fp8 wide {shape}")


def test_gemm_into_strided_output(snip):
    X = inputs.normal_bf16((128, 256), 1.0, 4, 1)
    W = inputs.normal_bf16((64, 256), 1.0, 4, 2)
    a = snip.quantize_nvfp4(X.cuda(), layout=snip.MMA)
    b = snip.quantize_nvfp4(W.cuda(), layout=snip.MMA)
    out = torch.full((128, 96), 7.0, device="cuda")
    snip.gemm(snip.NVFP4, a, b, 128, 64, 256, out=out[:, :64])
    o = out.cpu().numpy()
    assert np.all(o[:, 64:] == 7.0)                        # nothing written past N
    gemm_close(o[:, :64], oracle.gemm_tn(oracle.quantize_nvfp4(X).dequant(), oracle.quantize_nvfp4(W).dequant()))


def test_rounding_overrides(snip):
    """A plan can switch the backward quantizations to round-to-nearest."""
    X, W, dY = inputs.single_linear_inputs(64, 128, 128, seed=2)
    plan = snip.Plan([snip.NVFP4], seed=1)
    for tag in (snip.TAG_DY_DGRAD, snip.TAG_WT_DGRAD, snip.TAG_DYT_WGRAD, snip.TAG_XT_WGRAD):
        plan.set_rounding(0, tag, snip.RTN)
    ws = snip.qlinear_workspace(plan, 0, 64, 128, 128)
    dX, dW = snip.qlinear_bwd(plan, 0, X.cuda(), W.cuda(), dY.cuda(), ws)
    gemm_close(dX.cpu().numpy(), oracle.qlinear_dgrad("nvfp4", dY, W, 0, 1, rnd_dy=0, rnd_wt=0))
    gemm_close(dW.cpu().numpy(), oracle.qlinear_wgrad("nvfp4", dY, X, 0, 1, rnd_dyt=0, rnd_xt=0))


def test_qlinear_argument_errors(snip):
    plan = snip.Plan([snip.NVFP4])
    X = torch.zeros((64, 120), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((128, 120), dtype=torch.bfloat16, device="cuda")
    ws = snip.Workspace(1 << 20)
    with pytest.raises(snip.SnipError) as e:
        snip.qlinear_fwd(plan, 0, X, W, ws)
    assert e.value.status == snip.SNIP_ERR_SHAPE
    X = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    small = snip.Workspace(1024)
    with pytest.raises(snip.SnipError) as e:
        snip.qlinear_fwd(plan, 0, X, W, small)
    assert e.value.status == snip.SNIP_ERR_WORKSPACE
    with pytest.raises(snip.SnipError):
        snip.qlinear_fwd(plan, 3, X, W, ws)


def _sampled_block_parity(snip, cfg, plan_fmts, seed=0, nrows=48):
    """Run the whole block on the GPU, compare sampled rows of Y, dX and dW
    (all columns) with the oracle in fp64."""
    rng = np.random.default_rng(1234)
    inp = inputs.block_inputs(cfg, seed=seed, device="cuda")
    plan = snip.Plan(plan_fmts, seed=seed)
    for j, lin in enumerate(cfg.linears):
        X = inp.X[lin.x_id]
        W, dY = inp.W[j], inp.dY[j]
        ws = snip.qlinear_workspace(plan, j, cfg.T, lin.K, lin.N)
        Y = snip.qlinear_fwd(plan, j, X, W, ws)
        dX, dW = snip.qlinear_bwd(plan, j, X, W, dY, ws)
        torch.cuda.synchronize()
        assert ws.status() == snip.SNIP_OK
        fmt = "nvfp4" if plan_fmts[j] == 1 else "fp8"
        Xc, Wc, dYc = X.cpu(), W.cpu(), dY.cpu()
        rows_t = np.sort(rng.choice(cfg.T, nrows, replace=False))
        rows_n = np.sort(rng.choice(lin.N, nrows, replace=False))
        xq = oracle.quantize(fmt, Xc, 0, 0, seed, oracle.stream_id(j, 0)).dequant()
        wq = oracle.quantize(fmt, Wc, 0, 0, seed, oracle.stream_id(j, 1)).dequant()
        gemm_close(Y[rows_t].cpu().numpy(), oracle.gemm_tn(xq, wq, rows_t), f"{lin.name} Y")
        del xq, wq
        dyq = oracle.quantize(fmt, dYc, 0, 1, seed, oracle.stream_id(j, 2)).dequant()
        wtq = oracle.quantize(fmt, Wc, 1, 1, seed, oracle.stream_id(j, 3)).dequant()
        gemm_close(dX[rows_t].cpu().numpy(), oracle.gemm_tn(dyq, wtq, rows_t), f"{lin.name} dX")
        del dyq, wtq
        dytq = oracle.quantize(fmt, dYc, 1, 1, seed, oracle.stream_id(j, 4)).dequant()
        xtq = oracle.quantize(fmt, Xc, 1, 1, seed, oracle.stream_id(j, 5)).dequant()
        gemm_close(dW[rows_n].cpu().numpy(), oracle.gemm_tn(dytq, xtq, rows_n), f"{lin.name} dW")
        del dytq, xtq, Y, dX, dW, ws


@pytest.mark.slow
def test_tinyllama_block_sampled(snip):
    cfg = inputs.TINYLLAMA
    _sampled_block_parity(snip, cfg, inputs.seeded_plan(cfg, cfg.fp4_target, seed=0))


@pytest.mark.parametrize("fmt,code", FMTS)
@pytest.mark.parametrize("shape", [(256, 512, 384), (2048, 512, 2560)])
def test_qlinear_nonfinite_inputs(snip, fmt, code, shape):
    """A non-finite element in X (forward) or dY (backward) raises SNIP_ERR_NONFINITE in the
    workspace status and makes that tensor's statistics NaN; after a reset the same workspace gives
    exactly the results of a fresh one (one-CTA and CTA-pair GEMM shapes)."""
    T, K, N = shape
    X, W, dY = (inputs.normal_bf16(s, sg, 55, i).cuda() for i, (s, sg) in
                enumerate([((T, K), 1.0), ((N, K), 0.02), ((T, N), 1e-3)]))
    plan = snip.Plan([code], seed=2)
    ws = snip.qlinear_workspace(plan, 0, T, K, N)
    st = torch.zeros((3, snip.STATS_NVALS), dtype=torch.float64, device="cuda")
    Xbad = X.clone()
    Xbad[T // 2, K // 3] = float("inf")
    snip.qlinear_fwd(plan, 0, Xbad, W, ws, stats=st[0:2])
    assert ws.status() == snip.SNIP_ERR_NONFINITE
    assert np.isnan(st[0].cpu().numpy()).all()
    ws.reset()
    dYbad = dY.clone()
    dYbad[T - 1, N - 1] = float("nan")
    snip.qlinear_bwd(plan, 0, X, W, dYbad, ws, stats=st[2])
    assert ws.status() == snip.SNIP_ERR_NONFINITE
    assert np.isnan(st[2].cpu().numpy()).all()
    ws.reset()
    Y = snip.qlinear_fwd(plan, 0, X, W, ws)
    dX, dW = snip.qlinear_bwd(plan, 0, X, W, dY, ws)
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK
    fresh = snip.qlinear_workspace(plan, 0, T, K, N)
    Y2 = snip.qlinear_fwd(plan, 0, X, W, fresh)
    dX2, dW2 = snip.qlinear_bwd(plan, 0, X, W, dY, fresh)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y2) and torch.equal(dX, dX2) and torch.equal(dW, dW2)
