"""Stream order under programmatic dependent launch.  The quantizer and GEMM
kernels are launched so that the next kernel on a stream may be scheduled
while the previous one ends; each must still wait for the work before it.
Here every library call reads a buffer that the launch just before it on the
same stream wrote -- a PyTorch kernel, or another library kernel -- with no
synchronisation in between, and the source of each step is overwritten with
different data right after, so a call that read early or late would see the
wrong tensor.  Results must equal the same calls on inputs prepared and
synchronised beforehand, bit for bit."""
import pytest
import torch

from sub_byte_mixed_gb300 import inputs
from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def snip():
    return need_gpu()


def _chain(snip, X, W, dst_x, dst_w, ws):
    """copy -> scales -> quantize (both operands, two formats) -> GEMM, all back to back on one stream."""
    dst_x.copy_(X)
    dst_w.copy_(W)
    sx = snip.tensor_scales(dst_x, ws=ws)
    sw = snip.tensor_scales(dst_w, ws=ws)
    a = snip.quantize_nvfp4(dst_x, rnd=1, seed=3, stream_id=1, g_in=sx[1:2], layout=snip.MMA, ws=ws)
    b = snip.quantize_nvfp4(dst_w, rnd=0, seed=3, stream_id=2, g_in=sw[1:2], layout=snip.MMA, ws=ws)
    ft = snip.quantize_fp8(dst_x, orient=snip.ALONG_ROWS, rnd=1, seed=3, stream_id=4, s_in=sx[2:3],
                           layout=snip.MMA, ws=ws)
    M, K = X.shape
    N = W.shape[0]
    D = snip.gemm(snip.NVFP4, a, b, M, N, K, ws=ws)
    dst_x.fill_(3.0)    # the next writer of the sources: a call that read late would see it
    dst_w.fill_(-2.0)
    return D, a.codes, a.scales, b.codes, ft.codes


@pytest.mark.parametrize("M,N,K", [(512, 768, 1024), (2048, 1536, 2048)])
def test_back_to_back_calls_read_what_the_previous_launch_wrote(snip, M, N, K):
    ws = snip.Workspace(snip.snip_quantize_workspace_size(0, 0))
    dst_x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dst_w = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    runs = []
    for seed in (11, 12, 13):
        X = inputs.normal_bf16((M, K), 1.0, seed, 1).cuda()
        W = inputs.normal_bf16((N, K), 0.02, seed, 2).cuda()
        torch.cuda.synchronize()
        runs.append((X, W, _chain(snip, X, W, dst_x, dst_w, ws)))   # no synchronisation between the calls
    torch.cuda.synchronize()
    assert ws.status() == snip.SNIP_OK
    for X, W, got in runs:
        # the reference: inputs ready and synchronised before every call
        ref_x, ref_w = X.clone(), W.clone()
        torch.cuda.synchronize()
        want = _chain(snip, ref_x, ref_w, ref_x.clone(), ref_w.clone(), ws)
        torch.cuda.synchronize()
        for g, w in zip(got, want):
            assert torch.equal(g, w)
