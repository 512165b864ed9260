"""Pins of the oracle's tensor-level steps: block and tensor scales on
hand-built blocks, orientation, round-to-nearest idempotence, stochastic
rounding statistics over seeds, brute-force GEMMs, and statistics special
cases.  Each test is chosen so that a plausible mistake (a dropped term, a
wrong sign or index, a transposed operand) fails it."""
import math

import numpy as np
import pytest
import torch

from sub_byte_mixed_gb300 import inputs


def bf16(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def test_block_scale_closed_form(oracle_lib):
    """Block 0 holds the tensor max 2688 (so g = 1); block j > 0 holds max 6*k
    for an E4M3 value k, so its scale code is exactly k's code."""
    ks = [448.0, 1.0, 0.5, 1.5, 2.0 ** -6, 2.0 ** -9 * 3, 12.0, 0.0]
    row = np.zeros(16 * len(ks), dtype=np.float32)
    row[0] = 2688.0
    for j, k in enumerate(ks[1:], start=1):
        row[16 * j + 3] = 6.0 * k
        row[16 * j + 4] = -3.0 * k
    q = oracle_lib.quantize_nvfp4(bf16(row[None, :]))
    assert q.g == 1.0
    for j, k in enumerate(ks):
        assert oracle_lib.e4m3_value(q.scales[0, j]) == k, (j, k)
    xh = q.dequant()[0]
    # elements on the grid of their block come back exactly
    np.testing.assert_array_equal(xh, row.astype(np.float64))


def test_global_scale_definition(oracle_lib):
    x = bf16([[0.0] * 15 + [-5.0]])
    q = oracle_lib.quantize_nvfp4(x)
    assert q.g == np.float32(5.0) / np.float32(2688.0)
    z = oracle_lib.quantize_nvfp4(bf16(np.zeros((2, 32))))
    assert z.g == 1.0 and not z.codes.any() and not z.scales.any()
    f = oracle_lib.quantize_fp8(bf16([[0.5, -7.0, 1.0, 0.0]]))
    assert f.s == np.float32(7.0) / np.float32(448.0)


def test_element_codes_and_packing(oracle_lib):
    """g = 1, block scale 1: elements map to their own codes; byte j packs
    element 2j in the low nibble; negative zero keeps its sign (R4)."""
    vals = [6.0, 4.0, 3.0, 2.0, 1.5, 1.0, 0.5, 0.0, -6.0, -4.0, -3.0, -2.0, -1.5, -1.0, -0.5, -0.0]
    blk0 = np.zeros(16, dtype=np.float32); blk0[0] = 2688.0
    x = np.concatenate([blk0, np.array(vals, dtype=np.float32)])[None, :]
    q = oracle_lib.quantize_nvfp4(bf16(x))
    assert q.g == 1.0 and q.scales[0, 1] == 0x38          # E4M3 1.0 = 0 0111 000
    codes = []
    for b in q.codes[0, 8:]:
        codes += [int(b) & 15, int(b) >> 4]
    assert codes == [7, 6, 5, 4, 3, 2, 1, 0, 15, 14, 13, 12, 11, 10, 9, 8]


def test_saturation_when_scale_rounds_down(oracle_lib):
    """A block max of 6*(1+1/32) with g = 1: t = 1.03125 rounds to scale 1.0,
    the max element's scaled value 6.1875 saturates to code 7 (R2)."""
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0] = 2688.0
    x[0, 16] = 6.1875
    q = oracle_lib.quantize_nvfp4(bf16(x))
    assert oracle_lib.e4m3_value(q.scales[0, 1]) == 1.0
    assert (int(q.codes[0, 8]) & 15) == 7


def test_column_orientation_is_row_orientation_of_transpose(oracle_lib):
    x = inputs.normal_bf16((48, 80), 1.0, seed=3, tensor_id=1)
    for fmt in ("nvfp4", "fp8"):
        a = oracle_lib.quantize(fmt, x, orient=1)
        b = oracle_lib.quantize(fmt, x.t().contiguous(), orient=0)
        np.testing.assert_array_equal(a.codes, b.codes)
        if fmt == "nvfp4":
            np.testing.assert_array_equal(a.scales, b.scales)
            assert a.g == b.g
        else:
            assert a.s == b.s


def test_column_orientation_sr_uses_source_index(oracle_lib):
    """With SR, element (r, c) of the transposed output draws the random bits
    of source index r*C + c: flipping one source element's bits only changes
    that output element (checked by comparing against a brute-force re-encode)."""
    x = inputs.normal_bf16((32, 16), 1.0, seed=5, tensor_id=2)
    q = oracle_lib.quantize_nvfp4(x, orient=1, rnd=1, seed=9, stream_id=4)
    qr = oracle_lib.quantize_nvfp4(x, orient=1, rnd=0)
    xb = x.float().numpy()
    g = q.g
    for c in range(16):
        for blk in range(2):
            s = oracle_lib.e4m3_value(q.scales[c, blk])
            p = np.float32(np.float32(s) * np.float32(g))
            inv = np.float32(1.0) / p
            for k in range(16):
                r = blk * 16 + k
                y = np.float32(abs(xb[r, c])) * inv
                u = oracle_lib.sr_bits(9, 4, r * 16 + c)
                mag = oracle_lib.e2m1_sr(float(y), u) if xb[r, c] != 0 else 0
                byte = q.codes[c, r // 2]
                code = (int(byte) >> 4) if r & 1 else (int(byte) & 15)
                assert (code & 7) == mag, (r, c)
    np.testing.assert_array_equal(q.scales, qr.scales)


def test_rtn_idempotent_with_fixed_power_of_two_scale(oracle_lib):
    """Q(deQ(Q(x))) == Q(x) bit-exactly with g held fixed (R10)."""
    x = inputs.normal_bf16((64, 128), 1.0, seed=1, tensor_id=7)
    g = 2.0 ** -8
    q1 = oracle_lib.quantize_nvfp4(x, g_in=g)
    xh = torch.from_numpy(q1.dequant().astype(np.float32))
    assert torch.equal(xh.to(torch.bfloat16).float(), xh)         # exact in bf16
    q2 = oracle_lib.quantize_nvfp4(xh.to(torch.bfloat16), g_in=g)
    np.testing.assert_array_equal(q1.codes, q2.codes)
    np.testing.assert_array_equal(q1.scales, q2.scales)
    f1 = oracle_lib.quantize_fp8(x, s_in=2.0 ** -6)
    fh = torch.from_numpy(f1.dequant().astype(np.float32)).to(torch.bfloat16)
    f2 = oracle_lib.quantize_fp8(fh, s_in=2.0 ** -6)
    np.testing.assert_array_equal(f1.codes, f2.codes)


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
def test_sr_unbiased_over_seeds(oracle_lib, fmt):
    """Mean over seeds of the SR-dequantized tensor converges to x: every
    element within 5 standard errors (SR variance bound (step/2)^2)."""
    x = inputs.normal_bf16((16, 64), 1.0, seed=2, tensor_id=3)
    S = 200
    acc = np.zeros((16, 64))
    for s in range(S):
        acc += oracle_lib.quantize(fmt, x, 0, 1, seed=s, stream_id=2).dequant()
    mean = acc / S
    xr = x.float().double().numpy()
    rtn = oracle_lib.quantize(fmt, x).dequant()
    step = np.maximum(np.abs(rtn - xr) * 2, 1e-12)      # >= distance to the far neighbour / 2
    if fmt == "nvfp4":
        q = oracle_lib.quantize_nvfp4(x)
        sdec = np.array([[oracle_lib.e4m3_value(v) for v in row] for row in q.scales]) * q.g
        step = np.repeat(sdec, 16, axis=1) * 2.0            # widest E2M1 step in units of x
    else:
        step = np.abs(xr) / 8 + 2.0 ** -9 * oracle_lib.quantize_fp8(x).s
    se = step / 2 / math.sqrt(S)
    assert np.all(np.abs(mean - xr) <= 5 * se + 1e-12)
    # and the bias is far below the round-to-nearest error on average
    assert np.abs(mean - xr).mean() < 0.5 * np.abs(rtn - xr).mean()


def test_sr_variance_closed_form(oracle_lib):
    """Mean over seeds of the SR squared error equals the analytic
    sum (hi-|y|)(|y|-lo) q^2 reported by the statistics (within 4%)."""
    x = inputs.normal_bf16((32, 64), 1.0, seed=4, tensor_id=4)
    S = 100
    xr = x.float().double().numpy()
    e4 = np.mean([((oracle_lib.quantize_nvfp4(x, 0, 1, s, 2).dequant() - xr) ** 2).sum() for s in range(S)])
    e8 = np.mean([((oracle_lib.quantize_fp8(x, 0, 1, s, 2).dequant() - xr) ** 2).sum() for s in range(S)])
    st = oracle_lib.quant_stats(x)
    assert abs(e4 / st["nvfp4_sr_var"] - 1) < 0.04
    assert abs(e8 / st["fp8_sr_var"] - 1) < 0.04


def _brute_gemm(a, b):
    M, K = a.shape
    N = b.shape[0]
    out = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            s = 0.0
            for k in range(K):
                s += a[i, k] * b[j, k]
            out[i, j] = s
    return out


def test_gemm_brute_force_tiny(oracle_lib):
    X, W, dY = inputs.single_linear_inputs(T=16, K=32, N=16, seed=11)
    for fmt in ("nvfp4", "fp8"):
        xq = oracle_lib.quantize(fmt, X).dequant()
        wq = oracle_lib.quantize(fmt, W).dequant()
        np.testing.assert_allclose(oracle_lib.gemm_tn(xq, wq), _brute_gemm(xq, wq), rtol=1e-13, atol=1e-15)
        Y = oracle_lib.qlinear_fwd(fmt, X, W)
        np.testing.assert_allclose(Y, _brute_gemm(xq, wq), rtol=1e-13, atol=1e-15)
        # sampled rows agree with the full product
        np.testing.assert_array_equal(oracle_lib.gemm_tn(xq, wq, rows=np.array([3, 0, 15])), Y[[3, 0, 15]])


def test_gemm_identity_passthrough(oracle_lib):
    X = inputs.normal_bf16((32, 64), 1.0, seed=12, tensor_id=1)
    W = torch.eye(64, dtype=torch.float32).mul(0.5).to(torch.bfloat16)
    xq = oracle_lib.quantize_nvfp4(X).dequant()
    wq = oracle_lib.quantize_nvfp4(W).dequant()
    d = np.diag(wq)
    assert np.all(d == d[0]) and abs(d[0] - 0.5) < 1e-6
    np.testing.assert_array_equal(oracle_lib.qlinear_fwd("nvfp4", X, W), xq * d[0])


@pytest.mark.parametrize("fmt,tol", [("nvfp4", 0.25), ("fp8", 0.08)])
def test_qlinear_approximates_full_precision(oracle_lib, fmt, tol):
    """Non-square shapes: forward, dgrad and wgrad approximate X W^T, dY W and
    dY^T X (a transposed operand or wrong orientation fails shape or error)."""
    X, W, dY = inputs.single_linear_inputs(T=64, K=96, N=48, seed=13)
    Xf, Wf, dYf = (t.double().numpy() for t in (X, W, dY))
    cases = [(oracle_lib.qlinear_fwd(fmt, X, W), Xf @ Wf.T),
             (oracle_lib.qlinear_dgrad(fmt, dY, W), dYf @ Wf),
             (oracle_lib.qlinear_wgrad(fmt, dY, X), dYf.T @ Xf)]
    for got, ref in cases:
        assert got.shape == ref.shape
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel < tol, rel


def test_stats_special_cases(oracle_lib):
    z = oracle_lib.quant_stats(bf16(np.zeros((4, 32))))
    assert z["sum_x2"] == 0 and z["nvfp4_err2"] == 0 and z["fp8_err2"] == 0
    assert z["ratio_nvfp4"] == math.inf and not z["below_sqrt3_nvfp4"]
    # a tensor on both grids (g = 1, block scale 1, FP8 scale 2688/448 = 6)
    row = np.zeros(32, dtype=np.float32)
    row[0] = 2688.0
    row[16:22] = [6.0, -3.0, 1.5, 0.0, 12.0 / 2, -6.0]
    on = oracle_lib.quant_stats(bf16(row[None, :]), want_block_err=True)
    assert on["nvfp4_err2"] == 0 and on["nvfp4_sr_var"] == 0
    assert not on["block_err_nvfp4"].any()
    assert on["sum_x2"] == float((row.astype(np.float64) ** 2).sum())
    assert on["amax"] == 2688.0 and on["count"] == 32


def test_stats_sum_and_errors_match_quantizers(oracle_lib):
    x = inputs.outlier_bf16(64, 256, seed=1, tensor_id=9, frac=0.01)
    st = oracle_lib.quant_stats(x, rnd=1, seed=3, stream_id=2, want_block_err=True)
    xr = x.double().numpy()
    assert st["sum_x2"] == pytest.approx((xr ** 2).sum(), rel=1e-12)
    q4 = oracle_lib.quantize_nvfp4(x, 0, 1, 3, 2, want_block_err=True)
    assert st["nvfp4_err2"] == pytest.approx(((q4.dequant() - xr) ** 2).sum(), rel=1e-12)
    np.testing.assert_allclose(st["block_err_nvfp4"], q4.block_sqerr, rtol=1e-12)
    q8 = oracle_lib.quantize_fp8(x, 0, 1, 3, 2)
    assert st["fp8_err2"] == pytest.approx(((q8.dequant() - xr) ** 2).sum(), rel=1e-12)
    be8 = ((q8.dequant() - xr) ** 2).reshape(64, 16, 16).sum(-1)
    np.testing.assert_allclose(st["block_err_fp8"], be8, rtol=1e-12)
    assert st["ratio_nvfp4"] == pytest.approx(math.sqrt(st["sum_x2"] / st["nvfp4_err2"]))


def test_sqrt3_flag_threshold(oracle_lib):
    """The flag fires exactly when ||A|| < sqrt(3) * noise ("FP4 all the way")."""
    raw = np.zeros(oracle_lib.ST_N)
    raw[oracle_lib.ST_SUM_X2] = 3.0 * 1.0001
    raw[oracle_lib.ST_NVFP4_ERR2] = 1.0
    raw[oracle_lib.ST_FP8_ERR2] = 1.0002
    d = oracle_lib.derive_stats(raw)
    assert not d["below_sqrt3_nvfp4"] and d["below_sqrt3_fp8"]


def test_nonfinite_rejected(oracle_lib):
    for bad in (float("inf"), float("nan"), -float("inf")):
        x = bf16([[1.0] * 15 + [bad]])
        with pytest.raises(oracle_lib.NonFiniteInput):
            oracle_lib.quantize_nvfp4(x)
        with pytest.raises(oracle_lib.NonFiniteInput):
            oracle_lib.quantize_fp8(x)
        with pytest.raises(oracle_lib.NonFiniteInput):
            oracle_lib.quant_stats(x)


def test_shape_rule(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.quantize_nvfp4(bf16(np.ones((2, 24))))
    with pytest.raises(ValueError):
        oracle_lib.quantize_nvfp4(bf16(np.ones((24, 32))), orient=1)


def test_output_row_selection_matches_full_quantization(oracle_lib):
    """Quantizing only some output rows gives exactly those rows of the full
    quantization (tensor scale from the whole tensor, random bits by each
    element's index in it), for every format, orientation and rounding."""
    g = torch.Generator().manual_seed(9)
    x = (torch.randn(64, 96, generator=g) * 2).to(torch.bfloat16)
    for fmt in ("nvfp4", "fp8", "mxfp4"):
        for orient, sel in ((0, np.array([63, 2, 17, 40])), (1, np.array([95, 0, 40, 41]))):
            for rnd in (oracle_lib.RTN, oracle_lib.SR):
                full = oracle_lib.quantize(fmt, x, orient, rnd, 3, 5)
                sub = oracle_lib.quantize(fmt, x, orient, rnd, 3, 5, rows=sel)
                np.testing.assert_array_equal(full.codes[sel], sub.codes)
                if fmt != "fp8":
                    np.testing.assert_array_equal(full.scales[sel], sub.scales)
                np.testing.assert_array_equal(full.dequant()[sel], sub.dequant())
