"""Pins of the oracle's FP8 E5M2 path (the gradient format of the NEXT-2
variant): decoding against torch.float8_e5m2, round-to-nearest-even with
saturation against torch's conversion, exhaustive stochastic-rounding
unbiasedness, the tensor scale, on-grid round trips and orientation."""
import math

import numpy as np
import pytest
import torch

import oracle


def test_e5m2_decode_matches_torch_float8():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e5m2_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c], (c, v, ref[c])
    assert oracle.e5m2_value(0x7B) == 57344.0


def _probe_values():
    vals = torch.arange(0x7C, dtype=torch.uint8).view(torch.float8_e5m2).double().numpy()
    mids = (vals[:-1] + vals[1:]) / 2
    m32 = mids.astype(np.float32)
    rng = np.random.default_rng(0)
    return np.concatenate([vals, mids, np.nextafter(m32, np.float32(np.inf)).astype(np.float64),
                           np.nextafter(m32, np.float32(0)).astype(np.float64),
                           [57344.0, 57345.0, 61439.0, 61440.0, 1e6, 2.0 ** -17, 2.0 ** -18, 3 * 2.0 ** -18, 0.0],
                           np.exp(rng.uniform(-20, 11, 3000))])


def test_e5m2_rtn_matches_torch_rne_with_saturation():
    t = _probe_values()
    ref = torch.from_numpy(t).clamp(max=57344.0).to(torch.float8_e5m2).view(torch.uint8).numpy()
    got = np.array([oracle.e5m2_rtn(float(v)) for v in t], dtype=np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(t[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


@pytest.mark.parametrize("y", [0.0, 1e-5, 6.1e-5, 0.3, 1.0, 1.3, 13.3, 1000.7, 40000.0, 57343.0, 57344.0, 6e4])
def test_e5m2_sr_unbiased_exhaustive(y):
    y32 = float(np.float32(y))
    outs = [oracle.e5m2_value(oracle.e5m2_sr(y32, u)) for u in range(65536)]
    mean = float(np.mean(outs))
    if y32 >= 57344.0:
        assert mean == 57344.0
        return
    vals = torch.arange(0x7C, dtype=torch.uint8).view(torch.float8_e5m2).double().numpy()
    lo, hi = vals[vals <= y32].max(), vals[vals > y32].min()
    assert set(outs) <= {lo, hi}
    assert abs(mean - y32) <= (hi - lo) * 2.0 ** -16 + 1e-15


def test_e5m2_tensor_quantization():
    g = torch.Generator().manual_seed(1)
    grid = torch.arange(0x7C, dtype=torch.uint8).view(torch.float8_e5m2).float()
    x = grid[torch.randint(0, 0x7C, (16, 48), generator=g)] * torch.where(torch.rand(16, 48, generator=g) < 0.5, -1.0, 1.0)
    x[0, 0] = 57344.0                               # amax 57344: s = 1, the grid round-trips
    q = oracle.quantize_e5m2(x.to(torch.bfloat16))
    assert q.s == 1.0
    np.testing.assert_array_equal(q.dequant(), x.to(torch.bfloat16).double().numpy())
    assert oracle.lib().oracle_e5m2_tensor_scale(0.0) == 1.0
    assert oracle.lib().oracle_e5m2_tensor_scale(57344.0 * 4) == 4.0
    y = (torch.randn(32, 64, generator=g) * 1e-3).to(torch.bfloat16)
    a = oracle.quantize_e5m2(y, orient=1, rnd=oracle.RTN)
    b = oracle.quantize_e5m2(y.t().contiguous(), orient=0, rnd=oracle.RTN)
    np.testing.assert_array_equal(a.codes, b.codes)
