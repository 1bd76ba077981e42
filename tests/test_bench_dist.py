"""The multi-rank path of bench.py, on CPU with two gloo ranks.

The fused sampling path does not shard across GPUs (one GPU per call), so
`bench.py --gpus N` runs N independent replicas: the only cross-rank steps are
the barrier and the max-over-ranks of the timed region, and the whole-job rate
is all ranks' tokens over the slowest rank's time.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        local_ms = 100.0 + 25.0 * rank  # rank 1 is the slow one
        mx = bench.reduce_max(local_ms, "cpu")
        rate = bench.replica_throughput(world, 64 * 1000, mx)
        q.put((rank, mx, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, mx, rate in got:
        assert mx == 125.0
        assert rate == pytest.approx(2 * 64 * 1000 / 0.125)


def test_reduce_max_without_process_group_is_identity():
    assert bench.reduce_max(3.5, "cpu") == 3.5
    assert bench.replica_throughput(1, 640, 10.0) == pytest.approx(64000.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, env=env, timeout=300)
    assert res.returncode == 0
    assert res.stdout.strip() == ""


def test_kernel_hash_ignores_comments_and_whitespace():
    """The traffic record is keyed by a hash of the kernel code: comment and
    whitespace edits keep it, code edits (including string literals) change it."""
    code = 'int f(int x) { return x + 1; }  // add one\n/* note */ const char *s = "a // b";\n'
    same = '// header\nint f(int x) {\n    return x + 1;  /* add\n one */\n}\nconst char *s = "a // b";'
    other = 'int f(int x) { return x + 2; }\nconst char *s = "a // b";\n'
    lit = 'int f(int x) { return x + 1; }\nconst char *s = "a // c";\n'
    assert bench._code_only(code) == bench._code_only(same)
    assert bench._code_only(code) != bench._code_only(other)
    assert bench._code_only(code) != bench._code_only(lit)
    assert "add one" not in bench._code_only(code)
    assert len(bench.kernel_source_hash()) == 16
