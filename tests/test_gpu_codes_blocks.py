"""Quantized operands at the full block sizes, bit for bit: for every linear of
the TinyLlama block (T = 4096), the 7B block (T = 8192) and the 70B block
(T = 16384) under the seeded mixed plan the bench runs (its FP4-FLOP target
for that block), each of the six quantizations the layer makes --
X, W (forward, round-to-nearest) and dY (dgrad, stochastic) as row blocks
through the statistics-fused kernel the bench step uses, W^T, dY^T, X^T
(stochastic) as column blocks -- with the layer's seed and stream ids, in
the MMA layout.  Sampled output rows of the codes and block scales, and the
tensor scale, equal the oracle's quantization of only those rows (its tensor
scale and random bits from the whole tensor)."""
import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import mma_codes_to_rowmajor, mma_scales_to_rowmajor, need_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SEED = 0
NROWS = 24
# (tag, tensor, orientation, rounding): the layer's six quantizations (rounding defaults of a plan)
QUANTS = [(oracle.TAG_X_FWD, "X", 0, 0), (oracle.TAG_W_FWD, "W", 0, 0), (oracle.TAG_DY_DGRAD, "dY", 0, 1),
          (oracle.TAG_WT_DGRAD, "W", 1, 1), (oracle.TAG_DYT_WGRAD, "dY", 1, 1), (oracle.TAG_XT_WGRAD, "X", 1, 1)]


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


def _check_block(snip, cfg):
    plan = inputs.seeded_plan(cfg, cfg.fp4_target, seed=SEED)
    rng = np.random.default_rng(77)
    for j, lin in enumerate(cfg.linears):
        nvfp4 = plan[j] == inputs.FMT_NVFP4
        fmt, name = (snip.NVFP4, "nvfp4") if nvfp4 else (snip.FP8, "fp8")
        X, W, dY = inputs.linear_inputs(cfg, j, seed=SEED, device="cuda")
        host = {"X": X.cpu(), "W": W.cpu(), "dY": dY.cpu()}
        dev = {"X": X, "W": W, "dY": dY}
        for tag, which, orient, rnd in QUANTS:
            sid = oracle.stream_id(j, tag)
            t = dev[which]
            rows_src, cols_src = t.shape
            orows, ocols = (rows_src, cols_src) if orient == 0 else (cols_src, rows_src)
            if orient == 0:   # row blocks: the fused statistics kernel of the layer path and the bench
                codes, scales, _ = snip.quantize_stats(fmt, t, rnd=rnd, seed=SEED, stream_id=sid)
            else:             # column blocks: the transposing kernel
                q = (snip.quantize_nvfp4 if nvfp4 else snip.quantize_fp8)(t, orient=snip.ALONG_ROWS, rnd=rnd,
                                                                         seed=SEED, stream_id=sid, layout=snip.MMA)
                codes, scales = q.codes, (q.scales if nvfp4 else None)
            ts = snip.tensor_scales(t)
            torch.cuda.synchronize()
            sel = np.sort(rng.choice(orows, NROWS, replace=False))
            ref = oracle.quantize(name, host[which], orient, rnd, SEED, sid, rows=sel)
            what = f"{cfg.name} {lin.name} {which} orient {orient}"
            _, c = mma_codes_to_rowmajor(codes, orows, ocols, fmt_nvfp4=nvfp4)
            np.testing.assert_array_equal(c[sel], ref.codes, err_msg=what)
            if nvfp4:
                _, sc = mma_scales_to_rowmajor(scales, orows, ocols)
                np.testing.assert_array_equal(sc[sel], ref.scales, err_msg=what)
                assert float(ts[1].cpu()) == float(ref.g), what
            else:
                assert float(ts[2].cpu()) == float(ref.s), what
            del codes, scales
        del X, W, dY, host, dev
        torch.cuda.empty_cache()


def test_tinyllama_block_codes(snip):
    _check_block(snip, inputs.TINYLLAMA)


def test_llama7b_block_codes(snip):
    _check_block(snip, inputs.LLAMA7B)


def test_llama70b_block_codes(snip):
    _check_block(snip, inputs.LLAMA70B)
