"""The benchmark step's two-stream schedule (quantizations on one stream, GEMMs
on another, operand buffers alternating between two sets by linear), issued
call by call and replayed from a captured CUDA graph, against the same calls
on one stream: Y, dX, dW and the statistics of every linear
must be identical, so no GEMM reads an operand before its quantization has
written it or after the next user of its buffer set has overwritten it.  The
step that computes a shared activation's scales, statistics and forward
quantization once (Q/K/V, Gate/Up), with the tensor scales of several linears
in one launch, gives exactly the results of the step that recomputes them for
every linear with one tensor-scale launch per linear, and so do the steps that
run the linears in another order, spread the GEMMs over one, two (linears
alternating) or three (forward, dgrad, wgrad) streams, and put the tensor-scale
passes on a stream of their own.  Every kernel is
launched with programmatic stream serialization, so this also checks that each
waits for the work it follows on its stream."""
import os
import sys

import pytest
import torch

from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


@pytest.mark.parametrize("plan_kind", ["mix", "nvfp4-b64"])
def test_two_stream_step_matches_one_stream(plan_kind):
    snip = need_gpu()
    import bench
    from sub_byte_mixed_gb300 import inputs
    cfg = inputs.TINYLLAMA
    plan = (inputs.seeded_plan(cfg, cfg.fp4_target, seed=0) if plan_kind == "mix"
            else inputs.all_plan(bench.FORMAT_OF_NAME[plan_kind]))
    unshared = bench.Step(cfg, plan, snip, "cuda", overlap=False, share_x=False, scales_per_launch=3)
    assert unshared.scale_launches == len(cfg.linears)
    unshared.run()
    torch.cuda.synchronize()
    assert unshared.status() == snip.SNIP_OK
    ref0 = ([y.clone() for y in unshared.Y], [d.clone() for d in unshared.dX], [w.clone() for w in unshared.dW],
            unshared.stats_host())
    assert unshared.launches_per_step > 0
    del unshared
    serial = bench.Step(cfg, plan, snip, "cuda", overlap=False, scales_per_launch=8)
    assert serial.scale_launches == 3   # Q alone; K, V, O (7 tensors); Gate, Up, Down (8)
    serial.run()
    torch.cuda.synchronize()
    assert serial.status() == snip.SNIP_OK
    ref = ([y.clone() for y in serial.Y], [d.clone() for d in serial.dX], [w.clone() for w in serial.dW],
           serial.raw.clone())
    for j in range(len(cfg.linears)):
        assert torch.equal(ref[0][j], ref0[0][j]) and torch.equal(ref[1][j], ref0[1][j]), ("shared X", j)
        assert torch.equal(ref[2][j], ref0[2][j]), ("shared X", j)
    assert (serial.stats_host() == ref0[3]).all()
    del serial
    over = bench.Step(cfg, plan, snip, "cuda", overlap=True, gemm_streams=1, scales_stream=False)
    for _ in range(2):   # the second step also reuses both buffer sets across the step boundary
        over.run()
    torch.cuda.synchronize()
    assert over.status() == snip.SNIP_OK
    for j in range(len(cfg.linears)):
        assert torch.equal(over.Y[j], ref[0][j]), ("Y", j)
        assert torch.equal(over.dX[j], ref[1][j]), ("dX", j)
        assert torch.equal(over.dW[j], ref[2][j]), ("dW", j)
    assert torch.equal(over.raw, ref[3])
    del over
    # the linears in another order (the shared activations' users no longer adjacent)
    order = ["Q", "Gate", "Up", "Down", "K", "V", "O"]
    moved = bench.Step(cfg, plan, snip, "cuda", overlap=True, order=order, gemm_streams=2, scales_stream=True)
    assert moved.order == order
    for _ in range(2):
        moved.run()
    torch.cuda.synchronize()
    assert moved.status() == snip.SNIP_OK
    for j in range(len(cfg.linears)):
        assert torch.equal(moved.Y[j], ref[0][j]) and torch.equal(moved.dX[j], ref[1][j]), ("order", j)
        assert torch.equal(moved.dW[j], ref[2][j]), ("order", j)
    assert torch.equal(moved.raw, ref[3])
    del moved
    # the same two-stream step captured once as a CUDA graph and replayed
    graph = bench.Step(cfg, plan, snip, "cuda", overlap=True, own_stream=True)
    graph.run()
    graph.capture()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert graph.status() == snip.SNIP_OK
    for j in range(len(cfg.linears)):
        assert torch.equal(graph.Y[j], ref[0][j]) and torch.equal(graph.dX[j], ref[1][j]), j
        assert torch.equal(graph.dW[j], ref[2][j]), j
    assert torch.equal(graph.raw, ref[3])
