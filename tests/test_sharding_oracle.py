"""The token-sharded data-parallel form of the quantized linear layer, checked
with the oracle on CPU ranks (gloo, world size 2): each rank holds a slice of
the tokens of X and dY (a multiple of 16 tokens) and the whole W.

  - one MAX all-reduce of the shards' amax gives every rank the tensor scales
    of the whole X and dY;
  - each shard draws the random bits of its elements' indices in the whole
    tensors, so its codes are exactly the unsharded quantization's rows
    (blocks along K or N) and columns (blocks along the tokens, which never
    straddle a shard boundary);
  - Y and dX are the unsharded products' rows; dW is one SUM all-reduce of the
    shards' partial products; SNIP's statistics are one SUM all-reduce of the
    shards' raw sums (amax: the MAX).

Every number is compared with the unsharded oracle on rank 0."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

T, K, N, LAYER, SEED = 64, 128, 96, 2, 11


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _q(fmt, x, orient, rnd, tag, scale, base):
    import oracle
    sid = oracle.stream_id(LAYER, tag)
    if fmt == "nvfp4":
        return oracle.quantize_nvfp4(x, orient, rnd, SEED, sid, g_in=scale, index_base=base)
    return oracle.quantize_fp8(x, orient, rnd, SEED, sid, s_in=scale, index_base=base)


def _scale(fmt, amax):
    import oracle
    return oracle.nvfp4_global_scale(amax) if fmt == "nvfp4" else oracle.fp8_tensor_scale(amax)


def _layer(fmt, X, W, dY, gx, gw, gdy, t0):
    """One rank's part of the layer: X, dY hold tokens t0.. of the whole tensors."""
    import oracle
    xq = _q(fmt, X, 0, oracle.RTN, oracle.TAG_X_FWD, gx, t0 * K)
    wq = _q(fmt, W, 0, oracle.RTN, oracle.TAG_W_FWD, gw, 0)
    dyq = _q(fmt, dY, 0, oracle.SR, oracle.TAG_DY_DGRAD, gdy, t0 * N)
    wtq = _q(fmt, W, 1, oracle.SR, oracle.TAG_WT_DGRAD, gw, 0)
    dytq = _q(fmt, dY, 1, oracle.SR, oracle.TAG_DYT_WGRAD, gdy, t0 * N)
    xtq = _q(fmt, X, 1, oracle.SR, oracle.TAG_XT_WGRAD, gx, t0 * K)
    Y = oracle.gemm_tn(xq.dequant(), wq.dequant())
    dX = oracle.gemm_tn(dyq.dequant(), wtq.dequant())
    dW = oracle.gemm_tn(dytq.dequant(), xtq.dequant())
    return {"xq": xq, "dyq": dyq, "dytq": dytq, "xtq": xtq, "Y": Y, "dX": dX, "dW": dW}


def _rank_main(rank, world, port, fmt, out):
    import torch.distributed as dist
    import oracle
    from sub_byte_mixed_gb300 import inputs
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        X, W, dY = inputs.single_linear_inputs(T, K, N, seed=SEED)   # each rank keeps only its tokens
        t0, t1 = rank * T // world, (rank + 1) * T // world
        Xr, dYr = X[t0:t1].contiguous(), dY[t0:t1].contiguous()
        am = torch.tensor([oracle.amax(Xr), oracle.amax(dYr)], dtype=torch.float64)
        dist.all_reduce(am, op=dist.ReduceOp.MAX)
        gx, gdy, gw = _scale(fmt, float(am[0])), _scale(fmt, float(am[1])), _scale(fmt, oracle.amax(W))
        part = _layer(fmt, Xr, W, dYr, gx, gw, gdy, t0)
        dW = torch.from_numpy(part["dW"].copy())
        dist.all_reduce(dW, op=dist.ReduceOp.SUM)
        # SNIP's statistics of the shard of dY under dY's tensor scales and the dgrad rounding
        st = oracle.quant_stats(dYr, oracle.SR, SEED, oracle.stream_id(LAYER, oracle.TAG_DY_DGRAD),
                                g_in=oracle.nvfp4_global_scale(float(am[1])),
                                s_in=oracle.fp8_tensor_scale(float(am[1])), index_base=t0 * N)["raw"]
        sums = torch.from_numpy(st.copy())
        amax_st = sums[oracle.ST_AMAX].clone()
        dist.all_reduce(sums, op=dist.ReduceOp.SUM)
        dist.all_reduce(amax_st, op=dist.ReduceOp.MAX)
        sums[oracle.ST_AMAX] = amax_st
        out.put((rank, t0, t1, part["xq"].codes, part["dyq"].codes, part["dytq"].codes, part["xtq"].codes,
                 part["Y"], part["dX"], dW.numpy(), sums.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
def test_token_sharded_layer_equals_unsharded(fmt):
    import oracle
    from sub_byte_mixed_gb300 import inputs
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, fmt, q)) for r in range(world)]
    for p in procs:
        p.start()
    parts = sorted((q.get(timeout=300) for _ in range(world)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    X, W, dY = inputs.single_linear_inputs(T, K, N, seed=SEED)
    full = _layer(fmt, X, W, dY, _scale(fmt, oracle.amax(X)), _scale(fmt, oracle.amax(W)),
                  _scale(fmt, oracle.amax(dY)), 0)
    bpe = 2 if fmt == "nvfp4" else 1   # elements per code byte
    for (_, t0, t1, xq, dyq, dytq, xtq, Y, dX, dW, sums) in parts:
        # codes: rows of the row-block operands, token columns of the column-block ones
        np.testing.assert_array_equal(xq, full["xq"].codes[t0:t1])
        np.testing.assert_array_equal(dyq, full["dyq"].codes[t0:t1])
        np.testing.assert_array_equal(dytq, full["dytq"].codes[:, t0 // bpe:t1 // bpe])
        np.testing.assert_array_equal(xtq, full["xtq"].codes[:, t0 // bpe:t1 // bpe])
        # products: the same dequantized rows (fp64; a BLAS may block a shard's rows differently)
        np.testing.assert_allclose(Y, full["Y"][t0:t1], rtol=1e-13, atol=1e-13 * np.abs(full["Y"]).max())
        np.testing.assert_allclose(dX, full["dX"][t0:t1], rtol=1e-13, atol=1e-13 * np.abs(full["dX"]).max())
        # dW: the shards' partial products summed (another order of the fp64 sum)
        np.testing.assert_allclose(dW, full["dW"], rtol=1e-12, atol=1e-12 * np.abs(full["dW"]).max())
        ref = oracle.quant_stats(dY, oracle.SR, SEED, oracle.stream_id(LAYER, oracle.TAG_DY_DGRAD))["raw"]
        np.testing.assert_allclose(sums[:7], ref[:7], rtol=1e-12)


def test_shard_bits_differ_without_the_index_base():
    """The index base matters: a shard quantized as a tensor of its own draws other random bits."""
    import oracle
    from sub_byte_mixed_gb300 import inputs
    _, _, dY = inputs.single_linear_inputs(T, K, N, seed=SEED)
    g = oracle.nvfp4_global_scale(oracle.amax(dY))
    full = oracle.quantize_nvfp4(dY, 0, oracle.SR, SEED, 5, g_in=g)
    half = dY[T // 2:].contiguous()
    good = oracle.quantize_nvfp4(half, 0, oracle.SR, SEED, 5, g_in=g, index_base=(T // 2) * N)
    bad = oracle.quantize_nvfp4(half, 0, oracle.SR, SEED, 5, g_in=g)
    np.testing.assert_array_equal(good.codes, full.codes[T // 2:])
    assert not np.array_equal(bad.codes, full.codes[T // 2:])
