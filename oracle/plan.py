"""Oracle for SNIP's layer-wise format selection.

TEST INFRASTRUCTURE ONLY (see the package docstring): only ``tests/`` may
import it; the product path never does and shares no code with it.

"SNIP: An Adaptive Mixed Precision Framework for Subbyte LLM Training",
Abstract and Figure 2: statistics gathered during training drive an integer
program that picks FP8 or FP4 per layer, minimising the summed quality loss
while a required share of the FLOPs (Figure 3's efficiency: the fraction of
FP4 FLOPs) runs in FP4.  The pages do not give the divergence formulas; the
cost of a format for a layer is read here as the relative squared
quantization error of the layer's three operand tensors (X, W, dY), each
under its own rounding, taken from the statistics pass.

The selection is written as its definition: every assignment of the two
formats to the layers is enumerated, those whose FP4 FLOPs reach the
requirement are kept, and the cheapest is returned (small layer counts
only).  The requirement counts FLOPs in units of the layers' greatest common
divisor U_l and asks for ceil(fraction * sum U_l - 1e-9) of them.
"""
from __future__ import annotations

import itertools
import math

FP8, NVFP4 = 0, 1
# raw statistics slots: ||A||^2, NVFP4 error^2, FP8 error^2
_SUM_X2, _ERR_NVFP4, _ERR_FP8 = 0, 1, 2


def proxy_costs(raw):
    """raw[layer][tensor][slot] for tensors X, W, dY -> (cost_fp8, cost_nvfp4),
    each the sum over the three tensors of error^2 / ||A||^2 (0 when ||A|| = 0)."""
    c8, c4 = [], []
    for layer in raw:
        s8 = s4 = 0.0
        for t in layer:
            x2 = float(t[_SUM_X2])
            if x2 > 0.0:
                s8 += float(t[_ERR_FP8]) / x2
                s4 += float(t[_ERR_NVFP4]) / x2
        c8.append(s8)
        c4.append(s4)
    return c8, c4


def required_units(flops, fraction):
    """(units per layer, required FP4 units) with FLOPs in units of their gcd."""
    ints = [int(f) for f in flops]
    g = 0
    for v in ints:
        g = math.gcd(g, v)
    g = g or 1
    units = [v // g for v in ints]
    need = math.ceil(fraction * float(sum(units)) - 1e-9)
    return units, min(max(need, 0), sum(units))


def select_brute_force(flops, cost_fp8, cost_nvfp4, fraction):
    """Cheapest assignment meeting the FP4 requirement, by enumeration.
    Returns (formats, total cost); formats is one optimal assignment."""
    n = len(flops)
    units, need = required_units(flops, fraction)
    best = None
    for fmts in itertools.product((FP8, NVFP4), repeat=n):
        if sum(u for u, f in zip(units, fmts) if f == NVFP4) < need:
            continue
        cost = sum(cost_nvfp4[i] if f == NVFP4 else cost_fp8[i] for i, f in enumerate(fmts))
        if best is None or cost < best[1]:
            best = (list(fmts), cost)
    return best
