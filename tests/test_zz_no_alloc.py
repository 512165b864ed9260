"""snip_tensor_scales_noalloc: the tensor-scales call for callers that cannot
allocate device memory at the point of the call (code under a framework
allocator that forbids raw cudaMalloc, a path where an allocation and the
device synchronisation it may bring are not allowed).  It keeps its scratch in a fixed device array inside the
library instead of a caller workspace.  Checked against snip_tensor_scales,
exactly (the scales are exact functions of the input), on two calls in a row
with different tensors, so a value left in the shared scratch by the first
call cannot leak into the second.  This file is collected last on purpose."""
import pytest
import torch

from sub_byte_mixed_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_noalloc_scales_match_workspace_version():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sub_byte_mixed_gb300 import build, snip
    build.build()
    snip.load()
    snip.snip_device_check()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [inputs.outlier_bf16(1040, 784, seed=3, tensor_id=7).cuda(),
             inputs.normal_bf16((4096, 2048), 1e-3, seed=4, tensor_id=8).cuda()]
    for x in cases:                                   # two calls in a row
        got = torch.full((3,), -1.0, dtype=torch.float32, device="cuda")
        snip.snip_tensor_scales_noalloc(x.data_ptr(), x.numel(), got.data_ptr(), stream)
        ref = snip.tensor_scales(x)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), (got, ref)
        assert got[0].item() == x.float().abs().max().item()
    with pytest.raises(snip.SnipError) as e:          # beyond the fixed scratch
        snip.snip_tensor_scales_noalloc(cases[0].data_ptr(), (1 << 30) + 1, got.data_ptr(), stream)
    assert e.value.status == snip.SNIP_ERR_SHAPE
