"""A tensor split by rows (tokens) across parts, each quantized with
snip_quantize_part under the whole tensor's scales and its first element's
index, gives exactly the whole tensor's codes and scales: the parts' output
rows (blocks along the columns) or output columns (blocks along the tokens)
of the whole quantization, in every operand format; with statistics, the
parts' raw sums add up to the whole tensor's.  One part is also checked
against the oracle's quantization of the same part at the same index."""
import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import STATS_REL, need_gpu

pytestmark = pytest.mark.gpu

T, C = 256, 512
CUTS = [0, 128, 256]


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


def _fmts(snip):
    # (format, elements per code byte, elements per scale byte or 0)
    return [(snip.NVFP4, 2, 16), (snip.FP8, 1, 0), (snip.MXFP4, 2, 32), (snip.FP8_E5M2, 1, 0),
            (snip.NVFP4_B64, 2, 16)]


@pytest.mark.parametrize("k", range(5))
@pytest.mark.parametrize("orient", [0, 1])
@pytest.mark.parametrize("rnd", [0, 1])
def test_parts_equal_whole(snip, k, orient, rnd):
    fmt, epb, eps = _fmts(snip)[k]
    x = inputs.normal_bf16((T, C), 1e-3, 30 + k, 1).cuda()
    sc = snip.tensor_scales(x)
    whole_c, whole_s, _ = snip.quantize_part(fmt, x, 0, sc, orient=orient, rnd=rnd, seed=3, stream_id=7)
    torch.cuda.synchronize()
    wc = whole_c.cpu().numpy()
    ws_ = whole_s.cpu().numpy() if whole_s is not None else None
    for t0, t1 in zip(CUTS[:-1], CUTS[1:]):
        c, s, _ = snip.quantize_part(fmt, x[t0:t1].contiguous(), t0 * C, sc, orient=orient, rnd=rnd, seed=3,
                                     stream_id=7)
        torch.cuda.synchronize()
        if orient == 0:
            np.testing.assert_array_equal(c.cpu().numpy(), wc.reshape(T, -1)[t0:t1].reshape(-1))
            if eps:
                np.testing.assert_array_equal(s.cpu().numpy(), ws_.reshape(T, -1)[t0:t1].reshape(-1))
        else:
            np.testing.assert_array_equal(c.cpu().numpy().reshape(C, -1), wc.reshape(C, -1)[:, t0 // epb:t1 // epb])
            if eps:
                np.testing.assert_array_equal(s.cpu().numpy().reshape(C, -1),
                                              ws_.reshape(C, -1)[:, t0 // eps:t1 // eps])


def test_whole_part_is_the_quantizer(snip):
    """index_base 0 over the whole tensor is the standalone quantizer with the same scale."""
    x = inputs.normal_bf16((T, C), 1.0, 40, 1).cuda()
    sc = snip.tensor_scales(x)
    c, s, _ = snip.quantize_part(snip.NVFP4, x, 0, sc, rnd=1, seed=2, stream_id=4)
    q = snip.quantize_nvfp4(x, rnd=1, seed=2, stream_id=4, g_in=sc[1:2])
    torch.cuda.synchronize()
    assert torch.equal(c, q.codes) and torch.equal(s, q.scales)


@pytest.mark.parametrize("orient", [0, 1])
def test_part_matches_oracle_at_its_index(snip, orient):
    x = inputs.normal_bf16((T, C), 1e-3, 41, 3)
    sc = snip.tensor_scales(x.cuda())
    g = float(sc[1].cpu())
    part = x[128:].contiguous()
    c, s, _ = snip.quantize_part(snip.NVFP4, part.cuda(), 128 * C, sc, orient=orient, rnd=1, seed=9, stream_id=12)
    torch.cuda.synchronize()
    ref = oracle.quantize_nvfp4(part, orient, 1, 9, 12, g_in=g, index_base=128 * C)
    np.testing.assert_array_equal(c.cpu().numpy().reshape(ref.codes.shape), ref.codes)
    np.testing.assert_array_equal(s.cpu().numpy().reshape(ref.scales.shape), ref.scales)


@pytest.mark.parametrize("k", [0, 1, 2])
@pytest.mark.parametrize("rnd", [0, 1])
def test_part_statistics_add_up(snip, k, rnd):
    fmt = _fmts(snip)[k][0]
    x = inputs.normal_bf16((T, C), 1e-3, 50 + k, 2).cuda()
    sc = snip.tensor_scales(x)
    _, _, whole = snip.quantize_part(fmt, x, 0, sc, rnd=rnd, seed=5, stream_id=6, stats=True)
    parts = [snip.quantize_part(fmt, x[t0:t1].contiguous(), t0 * C, sc, rnd=rnd, seed=5, stream_id=6, stats=True)[2]
             for t0, t1 in zip(CUTS[:-1], CUTS[1:])]
    torch.cuda.synchronize()
    w = whole.cpu().numpy()
    ps = [p.cpu().numpy() for p in parts]
    for j in range(5):   # sums of squares, errors and variances
        assert sum(p[j] for p in ps) == pytest.approx(w[j], rel=STATS_REL), j
    assert max(p[5] for p in ps) == w[5]            # amax
    assert sum(p[6] for p in ps) == w[6]            # element count
    ref = oracle.quant_stats(x.cpu(), rnd=rnd, seed=5, stream_id=6)["raw"]
    for j in range(7):
        assert w[j] == pytest.approx(ref[j], rel=STATS_REL, abs=1e-300), j


def test_part_argument_errors(snip):
    x = torch.zeros((32, 64), dtype=torch.bfloat16, device="cuda")
    sc = snip.tensor_scales(x)
    with pytest.raises(snip.SnipError) as e:
        snip.quantize_part(snip.NVFP4, x, 8, sc)                  # not a multiple of 16
    assert e.value.status == snip.SNIP_ERR_SHAPE
    with pytest.raises(snip.SnipError) as e:
        snip.quantize_part(snip.NVFP4, x, 0, sc, orient=1, stats=True)   # statistics: row blocks only
    assert e.value.status == snip.SNIP_ERR_INVALID_ARG
