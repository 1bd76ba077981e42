"""The oracle still reproduces its frozen answer on the tiny workload.

The fixture is written by tests/golden/make_golden.py, which calls only the
oracle; this guards the oracle's arithmetic against silent changes.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def test_tiny_golden():
    with open(os.path.join(HERE, "golden", "tiny_oracle.json")) as f:
        want = json.load(f)
    got = make_golden.compute()
    assert got["inputs_sha256"] == want["inputs_sha256"], (
        "the seeded tiny inputs changed (torch RNG?); regenerate the fixture")
    for key in ("idx", "best", "second", "logits_row0_first8", "logits_sum", "logprob",
                "xform_idx", "xform_best", "shard_idx", "shard_logmass", "group_idx", "group"):
        assert got[key] == want[key], key
