"""Seeded synthetic inputs for the quantized linear layer.

Holds only shapes, value distributions and per-layer precision plans of the
Llama-like workloads (SNIP, Figure 4: the seven linear layers Q, K, V, O, Gate,
Up, Down of a transformer block).  No quantization arithmetic lives here; both
the CUDA path's tests and the oracle's tests draw their inputs from this module.

Recipe: every tensor is ``N(0, 1)`` from ``torch.randn`` on a generator seeded
with ``(seed, tensor_id)``, multiplied by its sigma in fp32 and rounded to bf16
(round-to-nearest-even).  Activations X have sigma 1, weights 0.02, output
gradients dY 1e-3.  The outlier sweep tensor additionally scales a seeded set of
exactly ``floor(0.001 * n)`` distinct positions by 100.
"""
from __future__ import annotations

import itertools
from dataclasses import dataclass, field

import numpy as np
import torch

SIGMA_X, SIGMA_W, SIGMA_DY = 1.0, 0.02, 1e-3

LAYER_NAMES = ("Q", "K", "V", "O", "Gate", "Up", "Down")
FMT_FP8, FMT_NVFP4, FMT_MXFP4 = 0, 1, 2   # per-layer format codes of a plan
FMT_NVFP4_B32, FMT_NVFP4_B64, FMT_NVFP4_B128 = 5, 6, 7   # NVFP4 with 32 / 64 / 128 elements per scale
FP4_FORMATS = (FMT_NVFP4, FMT_MXFP4, FMT_NVFP4_B32, FMT_NVFP4_B64, FMT_NVFP4_B128)


def _gen(seed: int, tensor_id: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + int(tensor_id)) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def normal_bf16(shape, sigma: float, seed: int, tensor_id: int, device="cpu") -> torch.Tensor:
    """sigma * N(0,1) rounded to bf16, seeded by (seed, tensor_id)."""
    x = torch.randn(tuple(shape), generator=_gen(seed, tensor_id, device), dtype=torch.float32,
                    device=device)
    if sigma != 1.0:
        x.mul_(sigma)
    return x.to(torch.bfloat16)


def outlier_bf16(rows: int, cols: int, seed: int, tensor_id: int, frac: float = 0.001,
                 factor: float = 100.0, device="cpu") -> torch.Tensor:
    """N(0,1) tensor with floor(frac * n) distinct seeded positions scaled by ``factor``."""
    n = rows * cols
    x = torch.randn((n,), generator=_gen(seed, tensor_id, device), dtype=torch.float32, device=device)
    k = int(np.floor(frac * n))
    pos = torch.randperm(n, generator=_gen(seed, tensor_id + 0x5000, device), device=device)[:k]
    x[pos] *= factor
    return x.view(rows, cols).to(torch.bfloat16)


# ----------------------------------------------------------------------------- block shapes

@dataclass(frozen=True)
class Linear:
    name: str
    K: int          # in-features
    N: int          # out-features
    x_id: str       # which activation tensor feeds it (shared by Q/K/V and by Gate/Up)


@dataclass
class BlockConfig:
    name: str
    T: int
    hidden: int
    inter: int
    kv_out: int
    fp4_target: float | None = None     # FP4-FLOP fraction the seeded plan aims at
    linears: list = field(default_factory=list)

    def __post_init__(self):
        h, i, kv = self.hidden, self.inter, self.kv_out
        self.linears = [
            Linear("Q", h, h, "attn"), Linear("K", h, kv, "attn"), Linear("V", h, kv, "attn"),
            Linear("O", h, h, "o"), Linear("Gate", h, i, "mlp"), Linear("Up", h, i, "mlp"),
            Linear("Down", i, h, "down"),
        ]

    def flops_fwd_bwd(self) -> int:
        """6 T K N summed over the seven linears (forward + dgrad + wgrad)."""
        return sum(6 * self.T * l.K * l.N for l in self.linears)

    def fp4_flop_fraction(self, plan) -> float:
        tot = sum(l.K * l.N for l in self.linears)
        return sum(l.K * l.N for l, f in zip(self.linears, plan) if f in FP4_FORMATS) / tot


# TinyLlama-1B: hidden 2048, intermediate 5632, 32 heads / 4 KV heads (K,V out 256), 2 x 2048 tokens
TINYLLAMA = BlockConfig("tinyllama-1b-block", T=4096, hidden=2048, inter=5632, kv_out=256, fp4_target=0.5)
# Llama-7B: hidden 4096, intermediate 11008, 32 heads (K,V out 4096), 4 x 2048 tokens
LLAMA7B = BlockConfig("llama-7b-block", T=8192, hidden=4096, inter=11008, kv_out=4096, fp4_target=0.8)
# Llama-70B: hidden 8192, intermediate 28672, 64 heads / 8 KV heads (K,V out 1024), 8 x 2048 tokens
LLAMA70B = BlockConfig("llama-70b-block", T=16384, hidden=8192, inter=28672, kv_out=1024, fp4_target=0.8)

BLOCKS = {c.name: c for c in (TINYLLAMA, LLAMA7B, LLAMA70B)}


def seeded_plan(cfg: BlockConfig, target: float, seed: int = 0) -> list[int]:
    """Per-layer FP8/NVFP4 plan whose FP4-FLOP fraction is closest to ``target``.

    All 128 masks over (Q,K,V,O,Gate,Up,Down) are enumerated in increasing mask
    order; among those closest to the target (ties within 1e-12) one is picked
    by a seeded draw.  This stands in for SNIP's selection (its ILP is not
    printed on the pages) and for the random baseline of its Figure 3."""
    best, ties = None, []
    for mask in range(128):
        plan = [FMT_NVFP4 if (mask >> i) & 1 else FMT_FP8 for i in range(7)]
        d = abs(cfg.fp4_flop_fraction(plan) - target)
        if best is None or d < best - 1e-12:
            best, ties = d, [plan]
        elif abs(d - best) <= 1e-12:
            ties.append(plan)
    pick = int(np.random.default_rng(seed).integers(len(ties)))
    return ties[pick]


def all_plan(fmt: int) -> list[int]:
    return [fmt] * 7


@dataclass
class BlockInputs:
    X: dict            # activation tensors by x_id
    W: list            # weight per linear (N x K)
    dY: list           # output gradient per linear (T x N)


X_TENSOR_ID = {"attn": 1, "o": 2, "mlp": 3, "down": 4}


def block_inputs(cfg: BlockConfig, seed: int = 0, device="cpu") -> BlockInputs:
    """Inputs of one Llama-like block: shared activations for Q/K/V and for
    Gate/Up, own activations for O and Down, one weight and one dY per linear."""
    T, h, i = cfg.T, cfg.hidden, cfg.inter
    X = {k: normal_bf16((T, h if k != "down" else i), SIGMA_X, seed, tid, device) for k, tid in X_TENSOR_ID.items()}
    W = [normal_bf16((l.N, l.K), SIGMA_W, seed, 10 + j, device) for j, l in enumerate(cfg.linears)]
    dY = [normal_bf16((T, l.N), SIGMA_DY, seed, 20 + j, device) for j, l in enumerate(cfg.linears)]
    return BlockInputs(X, W, dY)


def linear_inputs(cfg: BlockConfig, j: int, seed: int = 0, device="cpu"):
    """(X, W, dY) of linear j of the block, the same tensors as block_inputs
    generates for it, without the other linears' tensors."""
    l = cfg.linears[j]
    return (normal_bf16((cfg.T, l.K), SIGMA_X, seed, X_TENSOR_ID[l.x_id], device),
            normal_bf16((l.N, l.K), SIGMA_W, seed, 10 + j, device),
            normal_bf16((cfg.T, l.N), SIGMA_DY, seed, 20 + j, device))


def single_linear_inputs(T=64, K=128, N=128, seed=0, device="cpu"):
    """The single-layer case: X ~ N(0,1), W ~ N(0, 0.02^2), dY ~ N(0, 1e-3^2)."""
    return (normal_bf16((T, K), SIGMA_X, seed, 1, device),
            normal_bf16((N, K), SIGMA_W, seed, 2, device),
            normal_bf16((T, N), SIGMA_DY, seed, 3, device))


def all_masks():
    return list(itertools.product((FMT_FP8, FMT_NVFP4), repeat=7))
