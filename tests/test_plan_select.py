"""SNIP's layer-wise format selection (host code in the C library) against the
oracle's enumeration of every assignment, plus the cases whose answer is
fixed by the definition: a zero target keeps every layer whose FP4 cost is
not lower in FP8, a full target puts every layer in FP4, the cost never falls
as the target rises, and the proxy costs are the relative errors of the
statistics pass."""
import numpy as np
import pytest

from oracle import plan as oplan
from sub_byte_mixed_gb300 import inputs, snip


def _check(flops, c8, c4, frac):
    fmts, got_frac, got_cost = snip.snip_plan_select(flops, c8, c4, frac)
    ref_fmts, ref_cost = oplan.select_brute_force(flops, list(c8), list(c4), frac)
    units, need = oplan.required_units(flops, frac)
    # the library's choice is feasible and as cheap as the best assignment
    assert sum(u for u, f in zip(units, fmts) if f == oplan.NVFP4) >= need
    cost = sum(c4[i] if f == oplan.NVFP4 else c8[i] for i, f in enumerate(fmts))
    assert cost == pytest.approx(got_cost, rel=1e-12, abs=1e-15)
    assert cost == pytest.approx(ref_cost, rel=1e-12, abs=1e-15)
    tot = float(sum(flops))
    f4 = sum(f for f, m in zip(flops, fmts) if m == oplan.NVFP4)
    assert got_frac == pytest.approx(f4 / tot if tot else 0.0, rel=1e-15)
    return fmts


@pytest.mark.parametrize("seed", range(12))
def test_matches_enumeration_random(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 13))
    flops = (rng.integers(1, 40, n) * 6 * 4096 * 64).astype(np.float64)
    c8 = rng.uniform(0.0, 1e-3, n)
    c4 = c8 + rng.uniform(-2e-4, 5e-3, n)      # FP4 usually costlier, sometimes not
    for frac in (0.0, 0.3, 0.5, 0.8, 0.95, 1.0):
        _check(flops, c8, c4, frac)


def test_llama_block_shapes_match_enumeration():
    for cfg in (inputs.TINYLLAMA, inputs.LLAMA7B, inputs.LLAMA70B):
        flops = np.array([6.0 * cfg.T * l.K * l.N for l in cfg.linears])
        rng = np.random.default_rng(7)
        c8 = rng.uniform(1e-4, 2e-4, len(flops))
        c4 = rng.uniform(1e-2, 3e-2, len(flops))
        for frac in (0.5, 0.8):
            _check(flops, c8, c4, frac)


def test_definition_cases():
    flops = [6.0 * 8192 * 4096 * 4096] * 4 + [6.0 * 8192 * 4096 * 11008] * 3
    c8 = [1.0] * 7
    c4 = [2.0, 3.0, 1.5, 4.0, 2.5, 2.2, 9.0]
    fmts, frac, cost = snip.snip_plan_select(flops, c8, c4, 0.0)
    assert fmts == [0] * 7 and frac == 0.0 and cost == 7.0
    fmts, frac, cost = snip.snip_plan_select(flops, c8, c4, 1.0)
    assert fmts == [1] * 7 and frac == 1.0 and cost == pytest.approx(sum(c4))
    # an FP4 cost below FP8's is taken even with no target
    fmts, _, _ = snip.snip_plan_select(flops, c8, [2.0, 0.5, 3.0, 3.0, 3.0, 3.0, 3.0], 0.0)
    assert fmts == [0, 1, 0, 0, 0, 0, 0]
    # the cost never falls as the target rises
    costs = [snip.snip_plan_select(flops, c8, c4, f)[2] for f in np.linspace(0, 1, 21)]
    assert all(b >= a - 1e-12 for a, b in zip(costs, costs[1:]))
    # no layers
    assert snip.snip_plan_select([], [], [], 0.5) == ([], 0.0, 0.0)


def test_zero_flop_layer_and_ties():
    fmts, frac, cost = snip.snip_plan_select([0.0, 6.0, 6.0], [1.0, 1.0, 1.0], [0.5, 2.0, 2.0], 0.5)
    assert fmts[0] == 1                       # free and cheaper in FP4
    assert sum(fmts[1:]) == 1 and cost == pytest.approx(0.5 + 2.0 + 1.0)
    # equal costs: FP8 wins the tie for a layer
    fmts, _, _ = snip.snip_plan_select([6.0, 6.0], [1.0, 1.0], [1.0, 1.0], 0.0)
    assert fmts == [0, 0]


def test_argument_errors():
    with pytest.raises(snip.SnipError):
        snip.snip_plan_select([6.0], [0.0], [0.0], 1.5)
    with pytest.raises(snip.SnipError):
        snip.snip_plan_select([6.5], [0.0], [0.0], 0.5)          # non-integral FLOPs
    with pytest.raises(snip.SnipError):
        snip.snip_plan_select([-6.0], [0.0], [0.0], 0.5)
    with pytest.raises(snip.SnipError):
        snip.snip_plan_select([6.0], [float("nan")], [0.0], 0.5)
    # a table larger than the limit: coprime FLOPs make the unit 1
    with pytest.raises(snip.SnipError) as e:
        snip.snip_plan_select([2.0 ** 40 + 1, 2.0 ** 40], [0.0, 0.0], [1.0, 1.0], 0.5)
    assert e.value.status == snip.SNIP_ERR_SHAPE


def test_proxy_costs_match_oracle():
    rng = np.random.default_rng(3)
    raw = rng.uniform(0.1, 10.0, (5, 3, snip.STATS_NVALS))
    raw[2, 1, 0] = 0.0                        # a zero tensor adds nothing
    c8, c4 = snip.snip_plan_costs(raw)
    r8, r4 = oplan.proxy_costs(raw)
    np.testing.assert_allclose(c8, r8, rtol=1e-15)
    np.testing.assert_allclose(c4, r4, rtol=1e-15)
    raw[1, 0, 1] = float("inf")
    with pytest.raises(snip.SnipError):
        snip.snip_plan_costs(raw)


def test_oracle_hand_cases():
    """The enumeration on cases worked by hand: layers of 1, 1 and 2 FLOP units
    with FP8 costs 1, 1, 1 and FP4 costs 2, 4, 3.  Half the FLOPs (2 units) in
    FP4: {layer 2} costs 1+1+3 = 5, {0, 1} costs 2+4+1 = 7, so layer 2 alone.
    Three units: {0, 2} costs 2+1+3 = 6, the cheapest set reaching 3."""
    f, c8, c4 = [6.0, 6.0, 12.0], [1.0, 1.0, 1.0], [2.0, 4.0, 3.0]
    assert oplan.required_units(f, 0.5) == ([1, 1, 2], 2)
    assert oplan.select_brute_force(f, c8, c4, 0.5) == ([0, 0, 1], 5.0)
    assert oplan.select_brute_force(f, c8, c4, 0.75) == ([1, 0, 1], 6.0)
    assert oplan.select_brute_force(f, c8, c4, 0.0) == ([0, 0, 0], 3.0)
    raw = [[[4.0, 1.0, 0.5], [2.0, 1.0, 0.25], [0.0, 3.0, 3.0]]]
    assert oplan.proxy_costs(raw) == ([0.5 / 4 + 0.25 / 2], [1.0 / 4 + 1.0 / 2])
