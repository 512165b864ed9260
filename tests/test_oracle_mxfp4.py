"""Pins of the oracle's MXFP4 path (OCP Microscaling Formats v1.0: 32 E2M1
values sharing one E8M0 power-of-two scale) against what the format fixes:
E8M0 values, the shared exponent's closed form, exact round trips of
on-grid blocks, saturation and ties, the error bound, orientation, and
unbiased stochastic rounding."""
import math

import numpy as np
import pytest
import torch

import oracle

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _bf16(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def test_e8m0_values():
    L = oracle.lib()
    for c in range(255):
        assert L.oracle_e8m0_value(c) == math.ldexp(1.0, c - 127)
    assert math.isnan(L.oracle_e8m0_value(255))


def test_shared_exponent_closed_form():
    L = oracle.lib()
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.lognormal(0, 20, 4000), [1.0, 2.0, 3.999, 4.0, 6.0, 7.0, 1e-40, 2.0 ** -126]])
    for v in _bf16(vals).float().numpy():
        v = float(v)
        if v == 0.0:
            continue
        m, e = math.frexp(v)              # v = m 2^e, m in [0.5, 1)
        assert L.oracle_mxfp4_shared_exp(v) == max(min(e - 1 - 2, 127), -127), v
    assert L.oracle_mxfp4_shared_exp(0.0) == -127


@pytest.mark.parametrize("s", [-20, -3, 0, 5])
def test_on_grid_blocks_round_trip(s):
    rng = np.random.default_rng(s + 50)
    blocks = rng.choice(E2M1, size=(4, 64)) * rng.choice([-1, 1], size=(4, 64))
    blocks[:, 0] = 6.0                     # block max 6 * 2^s: shared exponent s
    blocks[:, 32] = -6.0
    x = _bf16(blocks * 2.0 ** s)
    q = oracle.quantize_mxfp4(x)
    assert np.all(q.scales == s + 127)
    np.testing.assert_array_equal(q.dequant(), x.float().numpy())


def test_saturation_and_ties():
    row = np.zeros((1, 32), dtype=np.float32)
    row[0, :6] = [7.0, 5.0, 2.5, 0.25, 0.75, -7.0]   # amax 7: shared exponent 0
    q = oracle.quantize_mxfp4(_bf16(row))
    assert q.scales[0, 0] == 127
    np.testing.assert_array_equal(q.dequant()[0, :6], [6.0, 4.0, 2.0, 0.0, 1.0, -6.0])


def test_error_bound_and_orientation():
    g = torch.Generator().manual_seed(4)
    x = (torch.randn(64, 96, generator=g) * torch.exp(torch.randn(64, 96, generator=g) * 2)).to(torch.bfloat16)
    q = oracle.quantize_mxfp4(x)
    xf = x.float().numpy().astype(np.float64)
    scale = np.repeat(np.array([[math.ldexp(1.0, int(c) - 127) for c in r] for r in q.scales]), 32, axis=1)
    # unsaturated: half the grid step (<= 1 in units of the scale); saturated (|y| in (6, 8)): < 2
    assert np.all(np.abs(q.dequant() - xf) <= 2.0 * scale)
    qt = oracle.quantize_mxfp4(x, orient=1)
    q2 = oracle.quantize_mxfp4(x.t().contiguous())
    np.testing.assert_array_equal(qt.codes, q2.codes)
    np.testing.assert_array_equal(qt.scales, q2.scales)


def test_stochastic_rounding_unbiased():
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(8, 64, generator=g) * 3).to(torch.bfloat16)
    xf = x.float().numpy().astype(np.float64)
    n = 300
    acc = np.zeros_like(xf)
    for seed in range(n):
        acc += oracle.quantize_mxfp4(x, rnd=oracle.SR, seed=seed, stream_id=3).dequant()
    mean = acc / n
    # saturated elements are biased by definition (6 at the top); the others' SR error has
    # variance (hi-y)(y-lo) <= (step/2)^2 with step <= 2 in units of the block scale
    q0 = oracle.quantize_mxfp4(x)
    scale = np.repeat(np.array([[math.ldexp(1.0, int(c) - 127) for c in r] for r in q0.scales]), 32, axis=1)
    unsat = np.abs(xf) / scale < 6.0
    assert np.all(np.abs(mean - xf)[unsat] <= 5.0 * scale[unsat] / math.sqrt(n))
    # and the mean error over all unsaturated elements is far below one step
    assert abs(np.mean(((mean - xf) / scale)[unsat])) < 0.02
