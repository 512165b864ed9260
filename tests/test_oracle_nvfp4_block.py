"""Pins for the oracle's longer-block NVFP4 variant ("FP4 all the way", summary
page, Outline: the study varies the block size; B elements share one E4M3
scale under the tensor scale g).  Checked against things other than itself:
  - B = 16 is NVFP4: identical to the (separately pinned) NVFP4 quantizer;
  - E4M3 rounding is monotone, so a B-block's scale is the largest of its
    16-element sub-blocks' NVFP4 scales, and the sub-blocks holding that
    largest scale get exactly their NVFP4 codes (same scale, same bits);
  - with round-to-nearest a larger scale never gives a larger magnitude code;
  - a worked example by hand where the longer block represents the data exactly."""
import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs


def _mags(codes):
    return np.stack([codes & 7, (codes >> 4) & 7], -1).reshape(codes.shape[0], -1)


@pytest.mark.parametrize("orient", [0, 1])
@pytest.mark.parametrize("rnd", [0, 1])
def test_block16_is_nvfp4(orient, rnd):
    x = inputs.normal_bf16((64, 96), 1.0, 3, 1)
    a = oracle.quantize_nvfp4(x, orient, rnd, 5, 7)
    b = oracle.quantize_nvfp4_block(x, 16, orient, rnd, 5, 7)
    np.testing.assert_array_equal(a.codes, b.codes)
    np.testing.assert_array_equal(a.scales, b.scales)
    assert a.g == b.g


@pytest.mark.parametrize("block", [32, 64, 128])
@pytest.mark.parametrize("orient", [0, 1])
@pytest.mark.parametrize("rnd", [0, 1])
def test_block_scale_is_max_of_subblock_scales(block, orient, rnd):
    # rows with different magnitudes per 16-element sub-block, so the maxima differ inside a block
    x = inputs.normal_bf16((128, 256), 1.0, 4, 2).float()
    x = x * torch.exp(torch.randn(128, 16, generator=torch.Generator().manual_seed(9))).repeat_interleave(16, 1)
    x = x.to(torch.bfloat16)
    if orient == 1:
        x = x.t().contiguous()
    n16 = oracle.quantize_nvfp4(x, orient, rnd, 1, 2)
    nb = oracle.quantize_nvfp4_block(x, block, orient, rnd, 1, 2)
    r = block // 16
    sub = n16.scales.reshape(n16.scales.shape[0], -1, r)
    np.testing.assert_array_equal(nb.scales, sub.max(axis=2))
    # sub-blocks whose own scale is the block's: codes as NVFP4's
    c16 = n16.codes.reshape(n16.codes.shape[0], -1, 8)      # 8 bytes = one 16-element sub-block
    cb = nb.codes.reshape(nb.codes.shape[0], -1, 8)
    same = n16.scales == np.repeat(nb.scales, r, axis=1)
    assert same.any() and (~same).any()
    np.testing.assert_array_equal(cb[same], c16[same])
    if rnd == 0:
        assert np.all(_mags(nb.codes) <= _mags(n16.codes))


def test_worked_example_block32():
    # one 32-element block: sixteen 1.0 then sixteen 3.0, tensor scale g = 1.  Its maximum 3 gives
    # the E4M3 scale 3/6 = 0.5 (code 0x30), so 1.0 -> 2.0 (magnitude code 4) and 3.0 -> 6.0 (code 7):
    # the block is represented exactly.  NVFP4's own first sub-block (maximum 1, scale E4M3(1/6) =
    # 0.171875 = 1.375 x 2^-3, code 0x23) rounds 1/0.171875 = 5.82 to 6 (code 7) instead.
    x = torch.tensor([[1.0] * 16 + [3.0] * 16], dtype=torch.bfloat16)
    q = oracle.quantize_nvfp4_block(x, 32, g_in=1.0)
    assert q.scales.tolist() == [[0x30]]
    assert q.codes.tolist() == [[0x44] * 8 + [0x77] * 8]
    np.testing.assert_array_equal(q.dequant(), x.double().numpy())
    n = oracle.quantize_nvfp4(x, g_in=1.0)
    assert n.scales.tolist() == [[0x23, 0x30]]
    assert n.codes[0, :8].tolist() == [0x77] * 8


@pytest.mark.parametrize("block", [32, 64])
def test_round_to_nearest_error_bound(block):
    # RTN: every element within half a grid step (at its magnitude) of its value, unless it saturates
    x = inputs.normal_bf16((32, 256), 2.0, 6, 3)
    q = oracle.quantize_nvfp4_block(x, block)
    xd = x.double().numpy()
    err = np.abs(q.dequant() - xd)
    p = np.repeat(np.array([[oracle.e4m3_value(int(s)) for s in row] for row in q.scales]), block, axis=1) * q.g
    y = np.abs(xd) / p
    step = np.where(y < 2, 0.5, np.where(y < 4, 1.0, 2.0))
    assert np.all(err <= 0.5 * step * p * (1 + 1e-6) + 1e-30)


def test_shape_and_block_errors():
    x = inputs.normal_bf16((16, 48), 1.0, 7, 4)
    with pytest.raises(ValueError):
        oracle.quantize_nvfp4_block(x, 32)        # 48 columns: not whole 32-blocks
    with pytest.raises(ValueError):
        oracle.quantize_nvfp4_block(x, 24)        # not a power of two
