"""SNIP's statistics at the full sizes of the Llama-shaped blocks ("SNIP",
Abstract and Figure 2: statistics of activations, weights and gradients;
"FP4 all the way", Outline: the gradient norm against sqrt(3) x the
quantization noise), as the layer API computes them: fused into the row-block
quantizations of snip_qlinear_fwd (X and W, round to nearest) and
snip_qlinear_bwd (dY, stochastic rounding with the layer's stream).

The largest tensors of the 70B block (16384 x 28672 and 28672 x 8192, up to
470 M elements) exercise the fused kernel's fp32 per-thread partial sums over
thousands of elements before the fp64 cross-CTA reduction; one linear of each
smaller block is checked as well.  The oracle (single-threaded C) runs over
row slices of the tensor in a thread pool, each slice with the whole tensor's
scales (from the oracle's own amax) and its first element's index, so it
draws the whole tensor's random bits; the slices' fp64 sums add up to the
tensor's (the oracle's part form, pinned by the sharding tests).  Bound: 1e-4
relative on every sum."""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import STATS_REL, need_gpu

# raw statistics slots: sum x^2, NVFP4 err^2, FP8 err^2, NVFP4 SR variance, FP8 SR variance, amax, count
N_SUMS = 5


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


def oracle_stats_sliced(x_cpu, rnd, seed, stream_id, rows_per_slice=512):
    """The oracle's statistics of a whole bf16 tensor, computed over row slices
    in parallel threads (the oracle's C call releases the interpreter lock)."""
    bits = oracle._bits(x_cpu)
    rows, cols = bits.shape
    amax = oracle.amax(bits)
    g, s = oracle.nvfp4_global_scale(amax), oracle.fp8_tensor_scale(amax)
    # one small call first: the oracle fills its lookup tables on first use, single-threaded here
    oracle.quant_stats(bits[:1], rnd=rnd, seed=seed, stream_id=stream_id, g_in=g, s_in=s)

    def part(r0):
        r1 = min(rows, r0 + rows_per_slice)
        return oracle.quant_stats(bits[r0:r1], rnd=rnd, seed=seed, stream_id=stream_id, g_in=g, s_in=s,
                                  index_base=r0 * cols)["raw"]

    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        raws = list(ex.map(part, range(0, rows, rows_per_slice)))
    tot = np.zeros_like(raws[0])
    for r in raws:
        tot[:N_SUMS] += r[:N_SUMS]
        tot[6] += r[6]
    tot[5] = max(r[5] for r in raws)
    return tot


def check_stats(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    for k in range(N_SUMS):
        assert got[k] == pytest.approx(ref[k], rel=STATS_REL, abs=1e-300), (what, k, got[k], ref[k])
    assert got[5] == ref[5], (what, "amax", got[5], ref[5])
    assert got[6] == ref[6], (what, "count", got[6], ref[6])


def _layer_stats(snip, cfg, layer_name, which, fmts=None, seed=0):
    """Statistics of the named layer's tensors ("X", "W", "dY") from the layer
    API under the block's seeded plan, and the oracle's of the same tensors."""
    fmts = fmts or inputs.seeded_plan(cfg, cfg.fp4_target, seed=seed)
    j = [l.name for l in cfg.linears].index(layer_name)
    lin = cfg.linears[j]
    X, W, dY = inputs.linear_inputs(cfg, j, seed=seed, device="cuda")
    plan = snip.Plan(fmts, seed=seed)
    ws = snip.qlinear_workspace(plan, j, cfg.T, lin.K, lin.N)
    raw = torch.zeros((3, snip.STATS_NVALS), dtype=torch.float64, device="cuda")
    Y = snip.qlinear_fwd(plan, j, X, W, ws, stats=raw[0:2])
    del Y
    if "dY" in which:
        dX, dW = snip.qlinear_bwd(plan, j, X, W, dY, ws, stats=raw[2])
        del dX, dW
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK
    got = raw.cpu().numpy()
    out = []
    for name in which:
        t = {"X": X, "W": W, "dY": dY}[name]
        k = {"X": 0, "W": 1, "dY": 2}[name]
        rnd = 1 if name == "dY" else 0
        ref = oracle_stats_sliced(t.cpu(), rnd, seed, oracle.stream_id(j, k))
        out.append((f"{cfg.name} {layer_name} {name} {tuple(t.shape)}", got[k], ref))
    del X, W, dY, ws
    torch.cuda.empty_cache()
    return out


def test_sliced_oracle_equals_whole_oracle(oracle_lib):
    """The sliced oracle reproduces the one-call oracle (both roundings)."""
    x = inputs.outlier_bf16(1040, 784, seed=5, tensor_id=3)
    for rnd in (0, 1):
        whole = oracle.quant_stats(x, rnd=rnd, seed=7, stream_id=19)["raw"]
        sl = oracle_stats_sliced(x, rnd, 7, 19, rows_per_slice=96)
        for k in range(N_SUMS):
            assert sl[k] == pytest.approx(whole[k], rel=1e-12), (rnd, k)
        assert sl[5] == whole[5] and sl[6] == whole[6]


@pytest.mark.gpu
@pytest.mark.slow
@pytest.mark.parametrize("layer,which", [("Down", ("X",)), ("Gate", ("W", "dY"))])
def test_llama70b_block_statistics_full(snip, layer, which):
    for what, got, ref in _layer_stats(snip, inputs.LLAMA70B, layer, which):
        check_stats(got, ref, what)


@pytest.mark.gpu
@pytest.mark.slow
@pytest.mark.parametrize("cfg_name", ["tinyllama", "llama7b"])
def test_smaller_blocks_statistics_full(snip, cfg_name):
    cfg = {"tinyllama": inputs.TINYLLAMA, "llama7b": inputs.LLAMA7B}[cfg_name]
    for layer, which in (("Down", ("X", "dY")), ("Up", ("W",))):
        for what, got, ref in _layer_stats(snip, cfg, layer, which):
            check_stats(got, ref, what)
