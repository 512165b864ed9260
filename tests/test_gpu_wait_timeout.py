"""Failure detection without a GPU fault: the bounded wait that every GEMM
pipeline role uses gives up after its limit on a barrier phase that nothing
completes, raises the timeout bit of the workspace status word, and lets a
second waiting thread leave through the abort flag.  The host reads
SNIP_ERR_TIMEOUT, and the context stays usable: a quantization on the same
workspace afterwards is correct once the status is reset."""
import numpy as np
import pytest
import torch

import oracle
from sub_byte_mixed_gb300 import inputs
from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ms", [1, 20])
def test_bounded_wait_times_out_and_context_survives(limit_ms):
    snip = need_gpu()
    ws = snip.Workspace(snip.snip_quantize_workspace_size(0, 0))
    assert ws.status() == snip.SNIP_OK
    out = snip.wait_check(limit_ms * 1_000_000, ws)
    torch.cuda.synchronize()
    done0, done1, ns1 = (int(v) for v in out.cpu())
    assert done0 == 0 and done1 == 0                      # neither barrier phase completed
    assert ws.status() == snip.SNIP_ERR_TIMEOUT
    # the second thread left on the abort flag, well before its own (4x) limit
    assert limit_ms * 1e6 * 0.9 <= ns1 < 3 * limit_ms * 1e6
    ws.reset()
    assert ws.status() == snip.SNIP_OK
    x = inputs.normal_bf16((64, 256), 1.0, 5, 1)
    q = snip.quantize_nvfp4(x.cuda(), rnd=1, seed=2, stream_id=3, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK
    ref = oracle.quantize_nvfp4(x, rnd=1, seed=2, stream_id=3)
    np.testing.assert_array_equal(q.codes.cpu().numpy().reshape(ref.codes.shape), ref.codes)


def test_wait_check_arguments():
    snip = need_gpu()
    with pytest.raises(snip.SnipError) as e:
        snip.snip_wait_check(1000, None, snip.Workspace(256).ptr, 256, None)
    assert e.value.status == snip.SNIP_ERR_INVALID_ARG
