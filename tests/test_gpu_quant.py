"""GPU parity of the quantizers (amax, NVFP4 both orientations, FP8) against
the oracle: bit-exact codes, scales and tensor scales on identical seeded
inputs, for round-to-nearest and stochastic rounding, in both output layouts,
at sizes that span several tiles with ragged tails, plus edge cases."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import need_gpu, mma_codes_to_rowmajor, mma_scales_to_rowmajor

pytestmark = pytest.mark.gpu

SHAPES = [(64, 128), (48, 80), (272, 400), (1040, 784)]


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


def _x(shape, seed=0, tid=1, sigma=1.0):
    return inputs.normal_bf16(shape, sigma, seed, tid)


@pytest.mark.parametrize("shape", SHAPES + [(3, 16), (1, 8), (0, 32)])
def test_amax_exact(snip, shape):
    x = _x(shape, tid=5)
    got = snip.amax(x.cuda()).item()
    ref = float(x.float().abs().max()) if x.numel() else 0.0
    assert got == ref


@pytest.mark.parametrize("shape", [(64, 128), (1040, 784), (0, 16)])
def test_tensor_scales(snip, shape):
    x = _x(shape, tid=6)
    sc = snip.tensor_scales(x.cuda()).cpu().numpy()
    m = float(x.float().abs().max()) if x.numel() else 0.0
    assert sc[0] == m
    assert sc[1] == oracle.nvfp4_global_scale(m) and sc[2] == oracle.fp8_tensor_scale(m)


def test_tensor_scales_multi(snip):
    """One launch over tensors of very different sizes (empty, a ragged few,
    medium, large) gives each tensor the scales of its own pass; a
    non-finite tensor among them flags the status and NaNs only its own."""
    shapes = [(0, 16), (3, 16), (257, 96), (2048, 1024)]
    xs = [_x(sh, tid=20 + i) for i, sh in enumerate(shapes)]
    xs[1] = xs[1].float().mul(1e30).to(torch.bfloat16)          # a huge amax
    outs = [torch.full((3,), -1.0, device="cuda") for _ in xs]
    ws = snip.Workspace(snip.snip_quantize_workspace_size(0, 0))
    snip.tensor_scales_multi([x.cuda() for x in xs], outs, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK
    for x, o in zip(xs, outs):
        m = float(x.float().abs().max()) if x.numel() else 0.0
        sc = o.cpu().numpy()
        assert sc[0] == m and sc[1] == oracle.nvfp4_global_scale(m) and sc[2] == oracle.fp8_tensor_scale(m)
    bad = xs[2].clone()
    bad[100, 7] = float("inf")
    outs2 = [torch.zeros(3, device="cuda") for _ in range(3)]
    ws2 = snip.Workspace(snip.snip_quantize_workspace_size(0, 0))
    snip.tensor_scales_multi([xs[3].cuda(), bad.cuda(), xs[2].cuda()], outs2, ws=ws2)
    torch.cuda.synchronize()
    assert ws2.status() == snip.SNIP_ERR_NONFINITE
    assert np.isnan(outs2[1].cpu().numpy()).all()
    assert outs2[0].cpu().numpy()[0] == float(xs[3].float().abs().max())
    assert outs2[2].cpu().numpy()[0] == float(xs[2].float().abs().max())


def test_tensor_scales_multi_eight_tensors(snip):
    """The most tensors one launch takes (8: two linears' X, W and dY, one X shared), sizes from a
    few elements to a few million, each with the scales of its own pass; 0 or 9 tensors are
    SNIP_ERR_INVALID_ARG before anything is read."""
    shapes = [(5, 16), (4096, 1024), (1, 8), (2048, 2048), (257, 96), (3000, 1000), (64, 128), (1024, 4096)]
    xs = [_x(sh, tid=40 + i).cuda() for i, sh in enumerate(shapes)]
    outs = [torch.full((3,), -1.0, device="cuda") for _ in xs]
    ws = snip.Workspace(snip.snip_quantize_workspace_size(0, 0))
    snip.tensor_scales_multi(xs, outs, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK
    for x, o in zip(xs, outs):
        m = float(x.float().abs().max())
        sc = o.cpu().numpy()
        assert sc[0] == m and sc[1] == oracle.nvfp4_global_scale(m) and sc[2] == oracle.fp8_tensor_scale(m)
    L = snip.load()
    n = 9
    ptrs = (ctypes.c_void_p * n)(*([xs[0].data_ptr()] * n))
    ns = (ctypes.c_int64 * n)(*([xs[0].numel()] * n))
    op = (ctypes.c_void_p * n)(*([outs[0].data_ptr()] * n))
    st = torch.cuda.current_stream().cuda_stream
    for count in (0, 9):
        assert L.snip_tensor_scales_multi(count, ptrs, ns, op, ws.ptr, ws.nbytes, st) == snip.SNIP_ERR_INVALID_ARG


def test_precomputed_scales_match(snip):
    """Quantizing with g_in from snip_tensor_scales gives the same bits as
    letting the call compute the scale itself."""
    x = _x((272, 400), seed=9, tid=2).cuda()
    sc = snip.tensor_scales(x)
    for rnd in (0, 1):
        a = snip.quantize_nvfp4(x, rnd=rnd, seed=2, layout=snip.MMA)
        b = snip.quantize_nvfp4(x, rnd=rnd, seed=2, layout=snip.MMA, g_in=sc[1:2])
        assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales) and torch.equal(a.g, b.g)
        f = snip.quantize_fp8(x, orient=1, rnd=rnd, seed=2)
        h = snip.quantize_fp8(x, orient=1, rnd=rnd, seed=2, s_in=sc[2:3])
        assert torch.equal(f.codes, h.codes)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("orient", [0, 1])
@pytest.mark.parametrize("rnd", [0, 1])
def test_nvfp4_rowmajor_bit_exact(snip, shape, orient, rnd):
    x = _x(shape, seed=1, tid=2)
    q = snip.quantize_nvfp4(x.cuda(), orient=orient, rnd=rnd, seed=11, stream_id=3, want_block_err=True)
    ref = oracle.quantize_nvfp4(x, orient=orient, rnd=rnd, seed=11, stream_id=3, want_block_err=True)
    torch.cuda.synchronize()
    assert q.g.item() == ref.g
    np.testing.assert_array_equal(q.codes.cpu().numpy().reshape(ref.codes.shape), ref.codes)
    np.testing.assert_array_equal(q.scales.cpu().numpy().reshape(ref.scales.shape), ref.scales)
    np.testing.assert_allclose(q.block_err.cpu().numpy(), ref.block_sqerr, rtol=1e-4, atol=1e-30)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("orient", [0, 1])
@pytest.mark.parametrize("rnd", [0, 1])
def test_nvfp4_mma_layout_bit_exact(snip, shape, orient, rnd):
    x = _x(shape, seed=2, tid=3)
    q = snip.quantize_nvfp4(x.cuda(), orient=orient, rnd=rnd, seed=5, stream_id=9, layout=snip.MMA)
    ref = oracle.quantize_nvfp4(x, orient=orient, rnd=rnd, seed=5, stream_id=9)
    full_c, c = mma_codes_to_rowmajor(q.codes, ref.rows, ref.cols)
    full_s, s = mma_scales_to_rowmajor(q.scales, ref.rows, ref.cols)
    np.testing.assert_array_equal(c, ref.codes)
    np.testing.assert_array_equal(s, ref.scales)
    # padding holds zero codes and zero scales
    assert not full_c[ref.rows:].any() and not full_c[:, ref.cols // 2:].any()
    assert not full_s[ref.rows:].any() and not full_s[:, ref.cols // 16:].any()
    assert q.g.item() == ref.g


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("orient", [0, 1])
@pytest.mark.parametrize("rnd", [0, 1])
@pytest.mark.parametrize("layout", [0, 1])
def test_fp8_bit_exact(snip, shape, orient, rnd, layout):
    x = _x(shape, seed=3, tid=4)
    q = snip.quantize_fp8(x.cuda(), orient=orient, rnd=rnd, seed=8, stream_id=2, layout=layout)
    ref = oracle.quantize_fp8(x, orient=orient, rnd=rnd, seed=8, stream_id=2)
    if layout == 0:
        got = q.codes.cpu().numpy().reshape(ref.codes.shape)
    else:
        full, got = mma_codes_to_rowmajor(q.codes, ref.rows, ref.cols, fmt_nvfp4=False)
        assert not full[ref.rows:].any() and not full[:, ref.cols:].any()
    np.testing.assert_array_equal(got, ref.codes)
    assert q.s.item() == ref.s


def test_given_tensor_scale(snip):
    x = _x((64, 256), seed=4, tid=1)
    g = torch.tensor([2.0 ** -8], device="cuda")
    q = snip.quantize_nvfp4(x.cuda(), g_in=g)
    ref = oracle.quantize_nvfp4(x, g_in=2.0 ** -8)
    np.testing.assert_array_equal(q.codes.cpu().numpy().reshape(ref.codes.shape), ref.codes)
    np.testing.assert_array_equal(q.scales.cpu().numpy().reshape(ref.scales.shape), ref.scales)
    assert q.g.item() == 2.0 ** -8
    f = snip.quantize_fp8(x.cuda(), s_in=g)
    fr = oracle.quantize_fp8(x, s_in=2.0 ** -8)
    np.testing.assert_array_equal(f.codes.cpu().numpy().reshape(fr.codes.shape), fr.codes)


def test_special_values(snip):
    """Zeros and negative zeros, exact grid values, ties, saturation, tiny
    blocks whose scale underflows, and bf16 subnormals."""
    row = np.zeros(256, dtype=np.float32)
    row[0] = 2688.0
    row[16:32] = [6, 4, 3, 2, 1.5, 1, .5, 0, .25, .75, 1.25, 1.75, 2.5, 3.5, 5, 6.1875]
    row[32:48] = -row[16:32]
    row[48] = -0.0
    row[64:80] = 1e-5                      # scale underflows to 0 relative to g = 1
    row[80:96] = 2.0 ** -130               # bf16 subnormal
    row[96:112] = np.linspace(-3, 3, 16)
    x = torch.tensor(np.stack([row, row / 7, -row * 3]), dtype=torch.float32).to(torch.bfloat16)
    for orient in (0,):
        for rnd in (0, 1):
            q = snip.quantize_nvfp4(x.cuda(), orient=orient, rnd=rnd, seed=3, stream_id=1)
            ref = oracle.quantize_nvfp4(x, orient=orient, rnd=rnd, seed=3, stream_id=1)
            np.testing.assert_array_equal(q.codes.cpu().numpy().reshape(ref.codes.shape), ref.codes)
            np.testing.assert_array_equal(q.scales.cpu().numpy().reshape(ref.scales.shape), ref.scales)
            f = snip.quantize_fp8(x.cuda(), rnd=rnd, seed=3, stream_id=1)
            fr = oracle.quantize_fp8(x, rnd=rnd, seed=3, stream_id=1)
            np.testing.assert_array_equal(f.codes.cpu().numpy().reshape(fr.codes.shape), fr.codes)


def test_all_zero_and_tiny_tensors(snip):
    for x in (torch.zeros((32, 64), dtype=torch.bfloat16),
              torch.full((16, 32), 2.0 ** -133, dtype=torch.float32).to(torch.bfloat16)):
        for rnd in (0, 1):
            q = snip.quantize_nvfp4(x.cuda(), rnd=rnd)
            ref = oracle.quantize_nvfp4(x, rnd=rnd)
            assert q.g.item() == ref.g
            np.testing.assert_array_equal(q.codes.cpu().numpy().reshape(ref.codes.shape), ref.codes)
            np.testing.assert_array_equal(q.scales.cpu().numpy().reshape(ref.scales.shape), ref.scales)
            f = snip.quantize_fp8(x.cuda(), rnd=rnd)
            fr = oracle.quantize_fp8(x, rnd=rnd)
            np.testing.assert_array_equal(f.codes.cpu().numpy().reshape(fr.codes.shape), fr.codes)
            assert f.s.item() == fr.s


def test_e4m3_conversion_exhaustive_probe(snip):
    """The hardware E4M3 conversion used for block scales and FP8 RTN matches
    the oracle's nearest-even rule on every E4M3 midpoint and its neighbours:
    a tensor built so that y = x * (1/s) lands on those points (s = 1)."""
    vals = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    mids = ((vals[:-1].astype(np.float64) + vals[1:]) / 2)
    pts = np.concatenate([vals, mids])
    pts = pts[pts <= 448]
    b = torch.tensor(pts, dtype=torch.float32).to(torch.bfloat16)   # bf16-exact probes only
    b = b[b.float() == torch.tensor(pts, dtype=torch.float32)]
    n = (b.numel() // 16) * 16
    x = torch.cat([torch.tensor([448.0]), b[: n - 1].float()]).to(torch.bfloat16).view(1, -1)
    for rnd in (0, 1):
        f = snip.quantize_fp8(x.cuda(), rnd=rnd, seed=1)
        fr = oracle.quantize_fp8(x, rnd=rnd, seed=1)
        np.testing.assert_array_equal(f.codes.cpu().numpy().reshape(fr.codes.shape), fr.codes)


def test_nonfinite_sets_status(snip):
    ws = snip.Workspace(snip.snip_quantize_workspace_size(0, 0))
    x = torch.ones((16, 32), dtype=torch.bfloat16)
    x[3, 7] = float("inf")
    q = snip.quantize_nvfp4(x.cuda(), ws=ws)
    assert ws.status() == snip.SNIP_ERR_NONFINITE
    assert np.isnan(q.g.item())
    ws.reset()
    assert ws.status() == snip.SNIP_OK
    x[3, 7] = float("nan")
    snip.quantize_fp8(x.cuda(), ws=ws)
    assert ws.status() == snip.SNIP_ERR_NONFINITE


def test_argument_errors(snip):
    x = torch.zeros((16, 24), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(snip.SnipError) as e:
        snip.quantize_nvfp4(x)
    assert e.value.status == snip.SNIP_ERR_SHAPE
    y = torch.zeros(16 * 32 + 4, dtype=torch.bfloat16, device="cuda")[4:].view(16, 32)
    with pytest.raises(snip.SnipError) as e:
        snip.quantize_nvfp4(y)
    assert e.value.status == snip.SNIP_ERR_ALIGN
    with pytest.raises(snip.SnipError) as e:
        snip.snip_quantize_nvfp4(x.data_ptr(), 16, 32, 0, 0, 0, 0, None, 0, None, None, None, None, 0, 0, None)
    assert e.value.status == snip.SNIP_ERR_INVALID_ARG


@pytest.mark.slow
def test_outlier_sweep_full_size(snip):
    """8192 x 8192 bf16 with 0.1% outliers x100: NVFP4 RTN, NVFP4 SR seeds
    0..3 and FP8 RTN, bit-exact on every element."""
    x = inputs.outlier_bf16(8192, 8192, seed=0, tensor_id=100)
    xd = x.cuda()
    cases = [("nvfp4", 0, 0)] + [("nvfp4", 1, s) for s in range(4)] + [("fp8", 0, 0)]
    for fmt, rnd, seed in cases:
        if fmt == "nvfp4":
            q = snip.quantize_nvfp4(xd, rnd=rnd, seed=seed, stream_id=2)
            ref = oracle.quantize_nvfp4(x, rnd=rnd, seed=seed, stream_id=2)
            assert q.g.item() == ref.g
            assert np.array_equal(q.codes.cpu().numpy().reshape(ref.codes.shape), ref.codes), (fmt, rnd, seed)
            assert np.array_equal(q.scales.cpu().numpy().reshape(ref.scales.shape), ref.scales), (fmt, rnd, seed)
        else:
            q = snip.quantize_fp8(xd)
            ref = oracle.quantize_fp8(x)
            assert np.array_equal(q.codes.cpu().numpy().reshape(ref.codes.shape), ref.codes)


@pytest.mark.slow
@pytest.mark.parametrize("layout", [0, 1])
def test_column_blocks_of_a_very_wide_tensor(snip, layout):
    """16 rows x 4,194,368 columns quantized with blocks along the rows: over
    65535 x 64 output rows, which a two-dimensional grid of 64-row tiles could
    not cover.  NVFP4 (SR) and FP8 (SR); sampled output rows, the last ones
    included, bit-exact vs the oracle."""
    R, C = 16, 4194368
    x = inputs.normal_bf16((R, C), 1.0, 5, 31)
    xd = x.cuda()
    rng = np.random.default_rng(3)
    sel = np.unique(np.concatenate([rng.choice(C, 40, replace=False), np.arange(C - 8, C)]))
    q = snip.quantize_nvfp4(xd, orient=snip.ALONG_ROWS, rnd=snip.SR, seed=2, stream_id=9, layout=layout)
    ref = oracle.quantize_nvfp4(x, orient=1, rnd=1, seed=2, stream_id=9, rows=sel)
    if layout == snip.MMA:
        _, codes = mma_codes_to_rowmajor(q.codes, C, R)
        # the chunked scale image at the sampled rows only (the whole gather would need GBs of indices)
        s_all = q.scales.cpu().numpy()
        r = sel[:, None].astype(np.int64)
        kb = np.arange(R // 16)[None, :]
        ocp = 256
        off = ((r // 128) * (ocp // 64) + kb // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
        scales = np.zeros((C, R // 16), dtype=np.uint8)
        scales[sel] = s_all[off]
    else:
        codes = q.codes.cpu().numpy().reshape(C, R // 2)
        scales = q.scales.cpu().numpy().reshape(C, R // 16)
    np.testing.assert_array_equal(codes[sel], ref.codes)
    np.testing.assert_array_equal(scales[sel], ref.scales)
    assert q.g.item() == ref.g
    f = snip.quantize_fp8(xd, orient=snip.ALONG_ROWS, rnd=snip.SR, seed=2, stream_id=10, layout=layout)
    fref = oracle.quantize_fp8(x, orient=1, rnd=1, seed=2, stream_id=10, rows=sel)
    if layout == snip.MMA:
        _, fcodes = mma_codes_to_rowmajor(f.codes, C, R, fmt_nvfp4=False)
    else:
        fcodes = f.codes.cpu().numpy().reshape(C, R)
    np.testing.assert_array_equal(fcodes[sel], fref.codes)
