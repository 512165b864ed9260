"""Pins of the oracle's element formats, rounding rules and RNG against things
fixed outside the oracle: the E2M1 grid, torch's float8_e4m3fn conversions,
numpy's round-half-even, the Random123 known-answer vectors, and the
unbiasedness that defines stochastic rounding."""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


def test_e2m1_grid_matches_golden(oracle_lib):
    for code, val in _read_table("e2m1_grid.txt"):
        v = oracle_lib.e2m1_value(int(code))
        assert v == float(val) and math.copysign(1, v) == math.copysign(1, float(val)), code


def test_e4m3_decode_matches_torch_float8(oracle_lib):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle_lib.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c], (c, v, ref[c])
    assert oracle_lib.e4m3_value(0x7E) == 448.0
    assert math.isnan(oracle_lib.e4m3_value(0x7F)) and math.isnan(oracle_lib.e4m3_value(0xFF))


def _e4m3_probe_values():
    """Every finite E4M3 value, the midpoints between neighbours, one fp32 ulp
    either side of those, values past 448, the subnormal range, and a seeded
    log-uniform sample."""
    vals = np.array([float(torch.tensor(c, dtype=torch.uint8).view(torch.float8_e4m3fn).float())
                     for c in range(0x7F)], dtype=np.float64)
    mids = (vals[:-1] + vals[1:]) / 2
    probes = [vals, mids]
    m32 = mids.astype(np.float32)
    probes.append(np.nextafter(m32, np.float32(np.inf)).astype(np.float64))
    probes.append(np.nextafter(m32, np.float32(0)).astype(np.float64))
    probes.append(np.array([448.0, 449.0, 463.99, 464.0, 480.0, 1e4, 3e38, 2.0 ** -10, 2.0 ** -11,
                            1.5 * 2.0 ** -10, 2.0 ** -12, 1e-30, 0.0]))
    rng = np.random.default_rng(7)
    probes.append(np.exp(rng.uniform(np.log(2.0 ** -12), np.log(600.0), 4000)))
    return np.concatenate(probes).astype(np.float32)


def test_e4m3_rtn_matches_torch_rne_with_saturation(oracle_lib):
    t = _e4m3_probe_values()
    ref = torch.from_numpy(t).clamp(max=448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_lib.e4m3_rtn(float(v)) for v in t], dtype=np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(t[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


def _e2m1_rne_numpy(y: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even onto the E2M1 grid via numpy's half-even rounding:
    the grid spacing is 0.5 below 2, 1 on [2,4) and 2 from 4; saturate at 6."""
    y = y.astype(np.float64)
    spacing = np.where(y < 2, 0.5, np.where(y < 4, 1.0, 2.0))
    r = np.round(y / spacing) * spacing
    return np.minimum(r, 6.0)


def test_e2m1_rtn_matches_half_even_rounding_on_all_bf16(oracle_lib):
    bits = np.arange(0, 0x7F80, dtype=np.uint32)             # all finite non-negative bf16
    y = (bits << 16).view(np.float32)
    y = y[y <= 16.0]
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    extra = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(9))])
    y = np.concatenate([y, extra])
    ref = _e2m1_rne_numpy(y)
    got = np.array([oracle_lib.e2m1_value(oracle_lib.e2m1_rtn(float(v))) for v in y])
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(y[i]), got[i], ref[i]) for i in bad[:10]]


def test_e2m1_rtn_ties_to_even_code(oracle_lib):
    # midpoint -> the neighbour with the even code (R3)
    expect = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for y, v in expect.items():
        assert oracle_lib.e2m1_value(oracle_lib.e2m1_rtn(y)) == v, y


def _sr_mean_exhaustive(fn, value, y):
    ups = [value(fn(y, u)) for u in range(65536)]
    return float(np.mean(ups))


@pytest.mark.parametrize("y", [0.0, 0.1, 0.3, 0.5, 0.71, 1.0, 1.33, 1.9, 2.2, 2.99, 3.5, 4.7, 5.999, 6.0, 7.5])
def test_e2m1_sr_unbiased_exhaustive(oracle_lib, y):
    """Over all 2^16 random words, the mean of the rounded value equals y to
    within one step * 2^-16 (stochastic rounding preserves the expected
    value), and every outcome is one of the two neighbours."""
    y32 = float(np.float32(y))
    outs = {oracle_lib.e2m1_value(oracle_lib.e2m1_sr(y32, u)) for u in range(0, 65536, 97)}
    mean = _sr_mean_exhaustive(oracle_lib.e2m1_sr, oracle_lib.e2m1_value, y32)
    if y32 >= 6.0:
        assert mean == 6.0 and outs == {6.0}
        return
    grid = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    lo = max(g for g in grid if g <= y32)
    hi = min(g for g in grid if g > y32)
    assert outs <= {lo, hi}
    assert abs(mean - y32) <= (hi - lo) * 2.0 ** -16 + 1e-15


@pytest.mark.parametrize("y", [0.0, 0.0013, 0.0151, 0.3, 1.0, 1.07, 13.3, 100.1, 300.0, 447.9, 448.0, 500.0])
def test_e4m3_sr_unbiased_exhaustive(oracle_lib, y):
    y32 = float(np.float32(y))
    mean = _sr_mean_exhaustive(oracle_lib.e4m3_sr, oracle_lib.e4m3_value, y32)
    if y32 >= 448.0:
        assert mean == 448.0
        return
    vals = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    lo = vals[vals <= y32].max()
    hi = vals[vals > y32].min()
    assert abs(mean - y32) <= (hi - lo) * 2.0 ** -16 + 1e-15


def test_philox_known_answers(oracle_lib):
    rows = _read_table("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for r in rows:
        v = [int(t, 16) for t in r]
        assert oracle_lib.philox4x32_10(v[0:4], v[4:6]) == v[6:10]


def test_sr_bits_uniform(oracle_lib):
    """The 16-bit words drawn per element look uniform (chi-square over 16 bins)."""
    n = 1 << 14
    w = np.array([oracle_lib.sr_bits(1234, 5, e) for e in range(n)], dtype=np.int64)
    counts = np.bincount(w >> 12, minlength=16)
    chi2 = float(((counts - n / 16) ** 2 / (n / 16)).sum())
    assert chi2 < 50.0           # 15 dof: p ~ 1e-5
    # consecutive elements differ (no repeated halves)
    assert np.mean(w[1:] == w[:-1]) < 0.01
