"""snip_qlinear_fwd_multi: the forward of several layers that read one
activation (SNIP, Figure 4: Q, K, V read one X; Gate, Up another) with X's
scales, statistics and quantization computed once per group of layers that
quantize it alike.  Every output must be exactly what snip_qlinear_fwd gives
layer by layer (which the other tests check against the oracle): Y bit for
bit, the statistics of X and of every W identical; a layer whose X_FWD
rounding is stochastic keeps its own stream id."""
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


def _per_layer(snip, plan, layers, X, Ws):
    T, K = X.shape
    Ys, stats = [], []
    for l, W in zip(layers, Ws):
        ws = snip.qlinear_workspace(plan, l, T, K, W.shape[0])
        st = torch.zeros((2, snip.STATS_NVALS), dtype=torch.float64, device="cuda")
        Ys.append(snip.qlinear_fwd(plan, l, X, W, ws, stats=st))
        stats.append(st)
    torch.cuda.synchronize()
    return Ys, stats


@pytest.mark.parametrize("fmts,sr_layer,shape", [((1, 1, 1), None, None), ((0, 1, 0), None, None),
                                                 ((1, 2, 4, 5), None, None), ((1, 1, 0), 1, None),
                                                 ((1, 0), None, (272, 400, [400, 144]))])
def test_multi_forward_equals_per_layer(snip, fmts, sr_layer, shape):
    T, K = (256, 512) if shape is None else shape[:2]   # the last case: ragged T, K and N
    Ns = [512, 128, 256, 384][:len(fmts)] if shape is None else shape[2]
    X = inputs.normal_bf16((T, K), 1.0, 11, 1).cuda()
    Ws = [inputs.normal_bf16((n, K), 0.02, 11, 10 + i).cuda() for i, n in enumerate(Ns)]
    plan = snip.Plan(list(fmts) + [1], seed=5)          # one more layer that the call does not use
    if sr_layer is not None:
        plan.set_rounding(sr_layer, snip.TAG_X_FWD, snip.SR)
    layers = list(range(len(fmts)))
    ref_Y, ref_st = _per_layer(snip, plan, layers, X, Ws)
    ws = snip.qlinear_fwd_multi_workspace(plan, layers, T, K, Ns)
    sx = torch.zeros(snip.STATS_NVALS, dtype=torch.float64, device="cuda")
    sw = [torch.zeros(snip.STATS_NVALS, dtype=torch.float64, device="cuda") for _ in layers]
    Ys = snip.qlinear_fwd_multi(plan, layers, X, Ws, ws, stats_x=sx, stats_w=sw)
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK
    for i in layers:
        assert torch.equal(Ys[i], ref_Y[i]), i
        assert torch.equal(sw[i], ref_st[i][1]), i
    # X's statistics: those of the first layer's forward rounding
    assert torch.equal(sx, ref_st[0][0])


def test_multi_forward_against_oracle(snip):
    """One group on the 7B attention shapes cut to 512 tokens, against the oracle's fp64 products."""
    T, K = 512, 4096
    Ns = [4096, 4096, 4096]
    X = inputs.normal_bf16((T, K), 1.0, 12, 1)
    Ws = [inputs.normal_bf16((n, K), 0.02, 12, 10 + i) for i, n in enumerate(Ns)]
    plan = snip.Plan([1, 1, 1], seed=0)
    ws = snip.qlinear_fwd_multi_workspace(plan, [0, 1, 2], T, K, Ns)
    Ys = snip.qlinear_fwd_multi(plan, [0, 1, 2], X.cuda(), [w.cuda() for w in Ws], ws)
    torch.cuda.synchronize()
    xq = oracle.quantize("nvfp4", X, 0, 0, 0, 0).dequant()
    for i, W in enumerate(Ws):
        gemm_close(Ys[i].cpu().numpy(), oracle.gemm_tn(xq, oracle.quantize("nvfp4", W, 0, 0, 0, 8 * i + 1).dequant()),
                   f"Y{i}")


def test_multi_forward_argument_errors(snip):
    T, K = 64, 128
    X = torch.zeros((T, K), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((128, K), dtype=torch.bfloat16, device="cuda")
    plan = snip.Plan([1, 1], seed=0)
    ws = snip.qlinear_fwd_multi_workspace(plan, [0, 1], T, K, [128, 128])
    with pytest.raises(snip.SnipError) as e:
        snip.qlinear_fwd_multi(plan, [0, 0], X, [W, W], ws)            # a layer twice
    assert e.value.status == snip.SNIP_ERR_INVALID_ARG
    small = snip.Workspace(1024)
    with pytest.raises(snip.SnipError) as e:
        snip.qlinear_fwd_multi(plan, [0, 1], X, [W, W], small)
    assert e.value.status == snip.SNIP_ERR_WORKSPACE
    assert np.isfinite(ws.nbytes)
