"""SNIP's loop on the GPU: the statistics of one step of a TinyLlama-shaped
block (256 tokens) come out of snip_qlinear_fwd/bwd, snip_plan_costs turns
them into per-layer format costs and snip_plan_select picks the layer-wise
formats; the pick must be optimal under the oracle's own statistics and
enumeration (within the statistics' tolerance)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import plan as oplan
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu

STATS_REL = 1e-4


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


def test_plan_from_step_statistics(snip):
    cfg = inputs.BlockConfig("tinyllama-1b-block-256", T=256, hidden=2048, inter=5632, kv_out=256, fp4_target=0.5)
    inp = inputs.block_inputs(cfg, seed=3)
    seed = 11
    plan = snip.Plan([inputs.FMT_NVFP4] * len(cfg.linears), seed=seed)
    raw = torch.empty((len(cfg.linears), 3, snip.STATS_NVALS), dtype=torch.float64, device="cuda")
    ref = np.zeros((len(cfg.linears), 3, snip.STATS_NVALS))
    for j, l in enumerate(cfg.linears):
        X, W, dY = inp.X[l.x_id], inp.W[j], inp.dY[j]
        ws = snip.qlinear_workspace(plan, j, cfg.T, l.K, l.N)
        Xd, Wd = X.cuda(), W.cuda()
        snip.qlinear_fwd(plan, j, Xd, Wd, ws, stats=raw[j, :2])
        snip.qlinear_bwd(plan, j, Xd, Wd, dY.cuda(), ws, stats=raw[j, 2])
        torch.cuda.synchronize()
        assert ws.status() == snip.SNIP_OK
        ref[j, 0] = oracle.quant_stats(X)["raw"]
        ref[j, 1] = oracle.quant_stats(W)["raw"]
        ref[j, 2] = oracle.quant_stats(dY, rnd=1, seed=seed, stream_id=j * 8 + 2)["raw"]
    got = raw.cpu().numpy()
    np.testing.assert_allclose(got[..., :5], ref[..., :5], rtol=STATS_REL)

    c8, c4 = snip.snip_plan_costs(got)
    r8, r4 = oplan.proxy_costs(ref)
    np.testing.assert_allclose(c8, r8, rtol=STATS_REL)
    np.testing.assert_allclose(c4, r4, rtol=STATS_REL)
    flops = [6.0 * cfg.T * l.K * l.N for l in cfg.linears]
    fmts, frac, _ = snip.snip_plan_select(flops, c8, c4, cfg.fp4_target)
    assert frac >= cfg.fp4_target
    _, best = oplan.select_brute_force(flops, r8, r4, cfg.fp4_target)
    chosen = sum(r4[i] if f == oplan.NVFP4 else r8[i] for i, f in enumerate(fmts))
    assert chosen <= best * (1 + 2 * STATS_REL)
    # the selected plan runs: one layer of it through the quantized linear
    sel = snip.Plan(fmts, seed=seed)
    l = cfg.linears[0]
    Y = snip.qlinear_fwd(sel, 0, inp.X[l.x_id].cuda(), inp.W[0].cuda(), snip.qlinear_workspace(sel, 0, cfg.T, l.K, l.N))
    torch.cuda.synchronize()
    assert torch.isfinite(Y).all()
