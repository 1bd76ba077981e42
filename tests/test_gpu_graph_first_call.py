"""A library call captured into a CUDA graph before any direct call.

fs_sample_ex takes the caller's workspace, so it needs no warm-up call before
stream capture.  Run in a fresh child process (so that nothing of the library
has touched the device yet), its very first call is captured; replaying the
graph must give the direct call's sample, and the device status word (whose
address Stage 2 looks up once per context) must read clear.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
sys.path.insert(0, %r)
import torch
import exact_sampling_lm_gb300 as fs
torch.cuda.set_device(0)
g = torch.Generator(device="cpu").manual_seed(3)
# one CTA per batch tile, the multicast pair, the pair MMA
for B, V, D in ((24, 12011, 128), (256, 9000, 64), (256, 3000, 6144)):
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn((V, D), generator=g) * 0.1).to(torch.bfloat16).cuda()
    ws = fs.workspace(B, V, D)
    idx = torch.full((B,), -7, dtype=torch.int64, device="cuda")
    sc = torch.empty(B, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        fs.fs_sample_ex(H, W, temperature=0.9, seed=5, offset=6, out_idx=idx, out_score=sc, ws=ws)
    graph.replay()
    torch.cuda.synchronize()
    ref_i, ref_s, _ = fs.fs_sample_ex(H, W, temperature=0.9, seed=5, offset=6)
    torch.cuda.synchronize()
    assert torch.equal(idx, ref_i) and torch.equal(sc, ref_s), (idx[:8], ref_i[:8])
    assert fs.fs_get_device_status() == 0
    print("captured first call ok B=%%d" %% B)
''' % ROOT


def test_first_library_call_under_graph_capture():
    res = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True,
                         timeout=300)
    print(res.stdout)
    assert res.returncode == 0, res.stderr[-3000:]
    assert res.stdout.count("captured first call ok") == 3
