"""NEXT-3 in the layer path (SNIP, Figure 5: a layer's dX is the dY of the
layer before it).  snip_qlinear_bwd_chain writes the preceding layer's two
NVFP4 gradient operands in its dgrad epilogue, and snip_qlinear_bwd_q runs
that layer's backward from them.  Checked:
  - against the unfused library path (dX in fp32, rounded to bf16, quantized
    by the library's quantizer with the same delayed scale, rounding and
    stream ids): operands, amax, dW of the later layer and dX, dW of the
    preceding one bit for bit; snip_qlinear_bwd_q fed the library's own
    quantization of dY reproduces snip_qlinear_bwd;
  - against the oracle on operands whose dgrad product is exact in fp32
    (power-of-two tensor scales, every block scale 448): the operands bit for
    bit, and the preceding layer's dX and dW within the GEMM bounds."""
import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import gemm_close, mma_codes_to_rowmajor, mma_scales_to_rowmajor, need_gpu
from test_gpu_requant import _exact_operand

pytestmark = pytest.mark.gpu

SEED = 3
T, K1, N1 = 256, 512, 384        # the later layer (layer 1): X1 T x K1, W1 N1 x K1, dY1 T x N1
K0 = 320                         # the preceding layer (layer 0): X0 T x K0, W0 K1 x K0, its dY = dX1 (T x K1)
RAGGED = (272, 400, 208, 336)    # T, K1, N1, K0 off every tile boundary


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


def _lib_operands(snip, dY0, g):
    rows = snip.quantize_nvfp4(dY0, rnd=snip.SR, seed=SEED, stream_id=0 * 8 + 2, g_in=g, layout=snip.MMA)
    cols = snip.quantize_nvfp4(dY0, orient=snip.ALONG_ROWS, rnd=snip.SR, seed=SEED, stream_id=0 * 8 + 4, g_in=g,
                               layout=snip.MMA)
    return rows, cols


@pytest.mark.parametrize("dims", [(T, K1, N1, K0), RAGGED])
def test_chain_equals_unfused_library_path(snip, dims):
    T, K1, N1, K0 = dims
    X1 = inputs.normal_bf16((T, K1), 1.0, 21, 1).cuda()
    W1 = inputs.normal_bf16((N1, K1), 0.02, 21, 2).cuda()
    dY1 = inputs.normal_bf16((T, N1), 1e-3, 21, 3).cuda()
    X0 = inputs.normal_bf16((T, K0), 1.0, 21, 4).cuda()
    W0 = inputs.normal_bf16((K1, K0), 0.02, 21, 5).cuda()
    plan = snip.Plan([1, 1], seed=SEED)
    ws1 = snip.qlinear_workspace(plan, 1, T, K1, N1)
    ws0 = snip.qlinear_workspace(plan, 0, T, K0, K1)
    # unfused: fp32 dX1 -> bf16 -> the preceding layer's dY, quantized with a given (delayed) scale
    dX1, dW1 = snip.qlinear_bwd(plan, 1, X1, W1, dY1, ws1)
    dY0 = dX1.to(torch.bfloat16)
    g = snip.tensor_scales(dY0)[1:2].clone() * 0.9      # a delayed estimate: some values saturate
    rows, cols = _lib_operands(snip, dY0, g)
    dX0_ref, dW0_ref = snip.qlinear_bwd_q(plan, 0, X0, W0, rows, cols, ws0)
    torch.cuda.synchronize()
    # fused
    dX1c, dW1c, crows, ccols, amax = snip.qlinear_bwd_chain(plan, 1, 0, X1, W1, dY1, g, ws1, want_dx=True)
    dX0, dW0 = snip.qlinear_bwd_q(plan, 0, X0, W0, crows, ccols, ws0)
    torch.cuda.synchronize()
    assert ws0.status() == snip.SNIP_OK and ws1.status() == snip.SNIP_OK
    assert torch.equal(dX1c, dX1) and torch.equal(dW1c, dW1)
    assert torch.equal(crows.codes, rows.codes) and torch.equal(crows.scales, rows.scales)
    assert torch.equal(ccols.codes, cols.codes) and torch.equal(ccols.scales, cols.scales)
    assert float(amax.cpu()) == float(dY0.float().abs().max())
    assert torch.equal(dX0, dX0_ref) and torch.equal(dW0, dW0_ref)
    # without the fp32 dX the operands are the same
    none, dW1n, nrows, ncols, _ = snip.qlinear_bwd_chain(plan, 1, 0, X1, W1, dY1, g, ws1)
    torch.cuda.synchronize()
    assert none is None and torch.equal(dW1n, dW1)
    assert torch.equal(nrows.codes, rows.codes) and torch.equal(ncols.scales, cols.scales)


def test_bwd_q_reproduces_bwd(snip):
    """Fed the library's quantization of dY with dY's own tensor scale, snip_qlinear_bwd_q gives
    snip_qlinear_bwd's dX and dW exactly."""
    X0 = inputs.normal_bf16((T, K0), 1.0, 22, 4).cuda()
    W0 = inputs.normal_bf16((K1, K0), 0.02, 22, 5).cuda()
    dY0 = inputs.normal_bf16((T, K1), 1e-3, 22, 6).cuda()
    plan = snip.Plan([1, 1], seed=SEED)
    ws = snip.qlinear_workspace(plan, 0, T, K0, K1)
    dX_ref, dW_ref = snip.qlinear_bwd(plan, 0, X0, W0, dY0, ws)
    g = snip.tensor_scales(dY0)[1:2].clone()
    rows, cols = _lib_operands(snip, dY0, g)
    dX, dW = snip.qlinear_bwd_q(plan, 0, X0, W0, rows, cols, ws)
    torch.cuda.synchronize()
    assert torch.equal(dX, dX_ref) and torch.equal(dW, dW_ref)


def test_chain_against_oracle_on_exact_products(snip):
    dY1 = _exact_operand(1, T, N1, 31)                    # row blocks along N1, g = 2^-10
    W1 = _exact_operand(1, K1, N1, 32).t().contiguous()   # W1^T's row blocks (along N1) exact
    X1 = inputs.normal_bf16((T, K1), 1.0, 23, 1)
    X0 = inputs.normal_bf16((T, K0), 1.0, 23, 4)
    W0 = inputs.normal_bf16((K1, K0), 0.02, 23, 5)
    q = lambda a, o, sid: oracle.quantize("nvfp4", a, o, 1, SEED, sid).dequant()
    dX1_ref = oracle.gemm_tn(q(dY1, 0, 8 + 2), q(W1, 1, 8 + 3))
    assert np.array_equal(dX1_ref.astype(np.float32).astype(np.float64), dX1_ref)   # exact in fp32
    dY0 = torch.from_numpy(dX1_ref.astype(np.float32)).to(torch.bfloat16)
    gval = np.float32(0.9 * float(np.abs(dX1_ref).max()) / 2688.0)
    orows = oracle.quantize_nvfp4(dY0, orient=0, rnd=1, seed=SEED, stream_id=2, g_in=float(gval))
    ocols = oracle.quantize_nvfp4(dY0, orient=1, rnd=1, seed=SEED, stream_id=4, g_in=float(gval))
    plan = snip.Plan([1, 1], seed=SEED)
    ws1 = snip.qlinear_workspace(plan, 1, T, K1, N1)
    ws0 = snip.qlinear_workspace(plan, 0, T, K0, K1)
    g = torch.tensor([gval], dtype=torch.float32, device="cuda")
    dX1, _, rows, cols, amax = snip.qlinear_bwd_chain(plan, 1, 0, X1.cuda(), W1.cuda(), dY1.cuda(), g, ws1,
                                                      want_dx=True)
    dX0, dW0 = snip.qlinear_bwd_q(plan, 0, X0.cuda(), W0.cuda(), rows, cols, ws0)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dX1.cpu().numpy().astype(np.float64), dX1_ref)
    _, c = mma_codes_to_rowmajor(rows.codes, T, K1)
    _, sc = mma_scales_to_rowmajor(rows.scales, T, K1)
    np.testing.assert_array_equal(c, orows.codes)
    np.testing.assert_array_equal(sc, orows.scales)
    _, c = mma_codes_to_rowmajor(cols.codes, K1, T)
    _, sc = mma_scales_to_rowmajor(cols.scales, K1, T)
    np.testing.assert_array_equal(c, ocols.codes)
    np.testing.assert_array_equal(sc, ocols.scales)
    assert float(amax.cpu()) == float(dY0.float().abs().max())
    # the preceding layer's GEMMs on these operands
    gemm_close(dX0.cpu().numpy(), oracle.gemm_tn(orows.dequant(), q(W0, 1, 3)), "dX0")
    gemm_close(dW0.cpu().numpy(), oracle.gemm_tn(ocols.dequant(), q(X0, 1, 5)), "dW0")


def test_chain_argument_errors(snip):
    X = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    plan = snip.Plan([0, 1], seed=0)                     # layer 0 FP8: no NVFP4 operands to write
    ws = snip.qlinear_workspace(plan, 1, 64, 128, 128)
    with pytest.raises(snip.SnipError) as e:
        snip.qlinear_bwd_chain(plan, 1, 0, X, W, X, g, ws)
    assert e.value.status == snip.SNIP_ERR_INVALID_ARG
    nv = snip.quantize_nvfp4(X, layout=snip.MMA)
    with pytest.raises(snip.SnipError) as e:
        snip.qlinear_bwd_q(plan, 0, X, W, nv, nv, ws)    # an FP8 layer has no NVFP4 backward
    assert e.value.status == snip.SNIP_ERR_INVALID_ARG
