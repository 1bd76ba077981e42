"""Write tests/golden/tiny_oracle.json from the CPU oracle alone.

The fixture freezes the oracle's answer on the tiny workload (B=4, D=256,
V=4096, T=1.0; inputs from the seeded generators in ``workloads``) so that a
later change to the oracle's arithmetic shows up as a diff.  Run from the
repository root:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json")


def tiny_inputs():
    B = 4
    H = workloads.to_bits(workloads.make_hidden("tiny", B))
    W = workloads.to_bits(workloads.make_weights("tiny"))
    T = workloads.make_temperature("tiny", B)
    seed, offset = workloads.sampling_seed("tiny", B)
    return H, W, T, seed, offset


def input_digest(H, W):
    h = hashlib.sha256()
    h.update(H.tobytes())
    h.update(W.tobytes())
    return h.hexdigest()


def compute():
    H, W, T, seed, offset = tiny_inputs()
    idx, best, second, l64 = oracle.sample(H, W, T, seed, offset, want_logits=True)
    idx1, best1, second1, _ = oracle.sample(H, W, T, seed, offset + 1)
    return {
        "workload": "tiny B=4 D=256 V=4096 T=1.0",
        "inputs_sha256": input_digest(H, W),
        "seed": seed,
        "offsets": [offset, offset + 1],
        "idx": [idx.tolist(), idx1.tolist()],
        "best": [[float(x) for x in best], [float(x) for x in best1]],
        "second": [[float(x) for x in second], [float(x) for x in second1]],
        "logits_row0_first8": [float(x) for x in l64[0, :8]],
        "logits_sum": float(np.sum(l64)),
    }


if __name__ == "__main__":
    with open(OUT, "w") as f:
        json.dump(compute(), f, indent=1)
        f.write("\n")
    print("wrote", OUT)
