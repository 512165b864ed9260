"""Host threads: the library keeps a few process-wide caches (the driver's
tensor-map encoder, each kernel's raised shared-memory limit per device,
occupancy per kernel and device), filled on first use under a lock.  A
fresh process -- every cache empty -- runs quantizations and GEMMs (CTA
pair, one-CTA and FP8 paths) from four host threads at once, each on its
own CUDA stream with its own workspace; every result must equal the same
calls made one after another on one stream, bit for bit."""
import os
import subprocess
import sys

import pytest

from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, threading
sys.path.insert(0, ROOT)
import torch
from sub_byte_mixed_gb300 import build, snip, inputs
build.build()
snip.load()

SHAPES = [(2048, 2560, 512, snip.NVFP4), (512, 384, 256, snip.NVFP4), (2048, 2304, 384, snip.FP8), (256, 640, 256, snip.FP8)]

def job(i, M, N, K, fmt, stream, out):
    with torch.cuda.stream(stream):   # the current stream is per thread
        A = inputs.normal_bf16((M, K), 1.0, 60 + i, 1).cuda()
        B = inputs.normal_bf16((N, K), 0.02, 60 + i, 2).cuda()
        ws = snip.Workspace(snip.snip_quantize_workspace_size(0, 0))   # calls sharing a workspace must not overlap
        q = snip.quantize_nvfp4 if fmt == snip.NVFP4 else snip.quantize_fp8
        a = q(A, rnd=1, seed=i, stream_id=2, layout=snip.MMA, ws=ws)
        b = q(B, rnd=1, seed=i, stream_id=3, layout=snip.MMA, ws=ws)
        D = snip.gemm(fmt, a, b, M, N, K, ws=ws)
        stream.synchronize()
        out[i] = (a.codes.cpu(), b.codes.cpu(), D.cpu(), ws.status())

par = {}
streams = [torch.cuda.Stream() for _ in SHAPES]
threads = [threading.Thread(target=job, args=(i, *s, streams[i], par)) for i, s in enumerate(SHAPES)]
for t in threads: t.start()
for t in threads: t.join()
seq = {}
for i, s in enumerate(SHAPES):
    job(i, *s, torch.cuda.current_stream(), seq)
assert sorted(par) == sorted(seq) == list(range(len(SHAPES)))
for i in range(len(SHAPES)):
    for x, y in zip(par[i][:3], seq[i][:3]):
        assert torch.equal(x, y), i
    assert par[i][3] == seq[i][3] == snip.SNIP_OK
print("threads ok")
"""


def test_concurrent_host_threads_fresh_process():
    need_gpu()
    r = subprocess.run([sys.executable, "-c", CHILD.replace("ROOT", repr(ROOT))], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads ok" in r.stdout
