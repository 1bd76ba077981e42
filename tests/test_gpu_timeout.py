"""Failure detection without a GPU fault: Stage 1's bounded waits.

Every mbarrier wait in Stage 1 gives up after FS_WAIT_TIMEOUT_MS; the CTA
then sets the library's device error word, tells its other warps to stop,
frees its tensor memory and returns.  The test hook FS_FLAG_TEST_NO_LOADS
makes the loader issue nothing, so the first wait of every CTA runs out; the
call's Stage 2 must then return no token (index -1, NaN score) for every row,
the host must read FS_ERR_TIMEOUT, and the context must stay usable (once the
word is cleared, normal calls agree again).  Runs in a child process so that
the short timeout applies only there.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, time
sys.path.insert(0, %r)
import torch
import exact_sampling_lm_gb300 as fs
from exact_sampling_lm_gb300 import _lib
torch.cuda.set_device(0)
g = torch.Generator(device="cpu").manual_seed(1)
# one CTA per batch tile, the multicast pair, the pair MMA
for B, V, D in ((4, 4096, 256), (256, 20000, 64), (256, 3000, 6144)):
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn((V, D), generator=g) * 0.1).to(torch.bfloat16).cuda()
    ws = fs.workspace(B, V, D)
    t0 = time.time()
    # the whole call: Stage 1 gives up, and Stage 2 returns no token
    idx, score, _ = fs.fs_sample_ex(H, W, temperature=1.0, seed=1, offset=0, flags=0x100, ws=ws)
    torch.cuda.synchronize()
    dt = time.time() - t0
    assert torch.all(idx == -1) and torch.all(torch.isnan(score)), idx
    # while the word is set, every later Stage 2 refuses too (log-probability
    # form included), whatever its candidates hold
    i2, s2, lp = fs.fs_sample_logprob(H, W, temperature=1.0, seed=1, offset=0)
    torch.cuda.synchronize()
    assert torch.all(i2 == -1) and torch.all(torch.isnan(s2)) and torch.all(torch.isnan(lp))
    fs.fs_stage1(H, W, ws, temperature=1.0, seed=1, offset=0, flags=0x100)
    word = fs.fs_get_device_status()
    assert word == 1, word
    assert 0.1 < dt < 30, dt
    # the context still works and the word was cleared
    i1, s1 = fs.fs_sample(H, W, temperature=1.0, seed=1, offset=0)
    i2, s2, _ = fs.fs_sample_ex(H, W, temperature=1.0, seed=1, offset=0)
    torch.cuda.synchronize()
    assert torch.equal(i1, i2) and torch.equal(s1, s2)
    assert fs.fs_get_device_status() == 0
    print("timeout path ok B=%%d: %%.2f s" %% (B, dt))
''' % ROOT


def test_bounded_wait_expires_and_reports_timeout():
    env = dict(os.environ, FS_WAIT_TIMEOUT_MS="300")
    res = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True,
                         env=env, timeout=300)
    print(res.stdout)
    assert res.returncode == 0, res.stderr[-2000:]
    assert res.stdout.count("timeout path ok") == 3
