"""Parity of whole Llama-shaped blocks at their full sizes (7B: T = 8192,
70B: T = 16384) on sampled outputs: for every linear, a 48 x 48 submatrix of
each of Y, dX and dW (sampled rows and columns) against the oracle's fp64
products of only the quantized rows those entries need (tensor scales and
random bits from the whole tensors)."""
import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import gemm_close, need_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

FMT_NAMES = {0: "fp8", 1: "nvfp4", 2: "mxfp4"}
# forward (X, W, W^T, X^T) and gradient (dY, dY^T) operand formats of each layer format
FWD = {0: "fp8", 1: "nvfp4", 2: "mxfp4", 4: "fp8"}
GRAD = {0: "fp8", 1: "nvfp4", 2: "mxfp4", 4: "e5m2"}


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


def _block_sampled(snip, cfg, plan_fmts, seed=0, n=48):
    rng = np.random.default_rng(4321)
    inp = inputs.block_inputs(cfg, seed=seed, device="cuda")
    plan = snip.Plan(plan_fmts, seed=seed)
    for j, lin in enumerate(cfg.linears):
        X, W, dY = inp.X[lin.x_id], inp.W[j], inp.dY[j]
        ws = snip.qlinear_workspace(plan, j, cfg.T, lin.K, lin.N)
        Y = snip.qlinear_fwd(plan, j, X, W, ws)
        dX, dW = snip.qlinear_bwd(plan, j, X, W, dY, ws)
        torch.cuda.synchronize()
        assert ws.status() == snip.SNIP_OK
        t = np.sort(rng.choice(cfg.T, n, replace=False))
        nn = np.sort(rng.choice(lin.N, n, replace=False))
        kk = np.sort(rng.choice(lin.K, n, replace=False))
        ti, ni, ki = (torch.tensor(v, device="cuda") for v in (t, nn, kk))
        y = Y[ti][:, ni].cpu().numpy()
        dx = dX[ti][:, ki].cpu().numpy()
        dw = dW[ni][:, ki].cpu().numpy()
        del Y, dX, dW, ws
        ff, fg = FWD[plan_fmts[j]], GRAD[plan_fmts[j]]
        Xc, Wc, dYc = X.cpu(), W.cpu(), dY.cpu()
        q = lambda f, a, o, r, tag, rows: oracle.quantize(f, a, o, r, seed, oracle.stream_id(j, tag),
                                                          rows=rows).dequant()
        gemm_close(y, oracle.gemm_tn(q(ff, Xc, 0, 0, 0, t), q(ff, Wc, 0, 0, 1, nn)), f"{cfg.name} {lin.name} Y")
        gemm_close(dx, oracle.gemm_tn(q(fg, dYc, 0, 1, 2, t), q(ff, Wc, 1, 1, 3, kk)), f"{cfg.name} {lin.name} dX")
        gemm_close(dw, oracle.gemm_tn(q(fg, dYc, 1, 1, 4, nn), q(ff, Xc, 1, 1, 5, kk)), f"{cfg.name} {lin.name} dW")


@pytest.mark.parametrize("plan", ["mix", "nvfp4", "fp8", "mxfp4", "fp8-e5m2-grad"])
def test_llama7b_block_sampled(snip, plan):
    cfg = inputs.LLAMA7B
    fmts = (inputs.seeded_plan(cfg, cfg.fp4_target, seed=0) if plan == "mix" else
            inputs.all_plan({"nvfp4": inputs.FMT_NVFP4, "fp8": inputs.FMT_FP8, "mxfp4": inputs.FMT_MXFP4,
                             "fp8-e5m2-grad": 4}[plan]))
    _block_sampled(snip, cfg, fmts)


def test_llama70b_block_sampled(snip):
    cfg = inputs.LLAMA70B
    _block_sampled(snip, cfg, inputs.seeded_plan(cfg, cfg.fp4_target, seed=0))
