"""bench.py's launcher logic, on CPU.

The fused sampling path runs on one GPU: it does not shard, and Stage 1's
paired forms couple the two CTAs of a cluster (multicast W loads or one MMA
over both), which are kept to single-GPU runs.  So the GPU arm refuses --gpus N > 1 and torchrun worlds
larger than one (exit status 2, before touching a device), while the
reference arm (the CPU oracle) runs on rank 0 only and the other ranks exit
without work.
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _run(args, env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, env=env, timeout=300)


def test_gpu_arm_refuses_more_than_one_gpu():
    res = _run(["--gpus", "2", "--steps", "3", "--warmup", "3"], {})
    assert res.returncode == 2
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["n_gpus"] == 2 and "single-GPU" in line["refused"]


def test_gpu_arm_refuses_a_torchrun_world():
    for rank in ("0", "1"):
        res = _run(["--steps", "3", "--warmup", "3"],
                   {"RANK": rank, "WORLD_SIZE": "2", "LOCAL_RANK": rank})
        assert res.returncode == 2
        out = res.stdout.strip()
        assert (json.loads(out)["refused"] if rank == "0" else out == "")


def test_reference_arm_other_ranks_exit_without_work():
    res = _run(["--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3"],
               {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert res.returncode == 0
    assert res.stdout.strip() == ""


def test_both_arms_share_the_config_object():
    cfg = bench.bench_config("llama3_8b", 64, 128256)
    assert set(cfg) == {"workload", "global_batch", "per_gpu_batch", "parallelism", "l2"}
    assert cfg["global_batch"] == cfg["per_gpu_batch"] == 64


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
