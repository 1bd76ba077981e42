"""Write tests/golden/tiny_oracle.json from the CPU oracle alone.

The fixture freezes the oracle's answers on the tiny workload (B=4, D=256,
V=4096, T=1.0; inputs from the seeded generators in ``workloads``): the
sample at two offsets, the logits, the sampled token's log-probability, a
sample after bias / soft-cap / mask, three vocabulary shards and their
grouped combine.  A later change to the oracle's arithmetic shows up as a
diff.  Run from the
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


def extra_inputs(B, V):
    """Bias [V] in [-0.5, 0.5) and an allowed-token mask [B, ceil(V/32)], from
    PCG64's raw output (stable across numpy versions)."""
    raw = np.random.PCG64(2026).random_raw(V + B * ((V + 31) // 32))
    bias = ((raw[:V] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53 - 0.5).astype(np.float32)
    mask = (raw[V:] & np.uint64(0xFFFFFFFF)).astype(np.uint32).reshape(B, (V + 31) // 32)
    return bias, mask


def compute():
    H, W, T, seed, offset = tiny_inputs()
    idx, best, second, l32 = oracle.sample(H, W, T, seed, offset, want_logits=True)
    idx1, best1, second1, _ = oracle.sample(H, W, T, seed, offset + 1)
    # the wider rows: log-probability of the sample, transforms, shards and
    # the grouped combine, on the same inputs
    assert np.array_equal(l32, oracle.logits(H, W))
    lp = oracle.logprob(l32, T, idx)
    bias, mask = extra_inputs(*l32.shape)
    lx = oracle.transform_logits(l32, bias=bias, softcap=15.0, mask=mask)
    xidx, xbest, _, _ = oracle.sample_from_logits(lx, T, seed, offset)
    cuts = [(0, 1024), (1024, 3072), (3072, W.shape[0])]
    shards = [oracle.sample_shard(H, W[a:b], a, T, seed, offset) for a, b in cuts]
    gidx, grp = oracle.combine_groups(np.stack([s[0] for s in shards]),
                                      np.stack([s[2] for s in shards]), 777, offset)
    return {
        "workload": "tiny B=4 D=256 V=4096 T=1.0",
        "inputs_sha256": input_digest(H, W),
        "seed": seed,
        "offsets": [offset, offset + 1],
        "idx": [idx.tolist(), idx1.tolist()],
        "best": [[float(x) for x in best], [float(x) for x in best1]],
        "second": [[float(x) for x in second], [float(x) for x in second1]],
        "logits_row0_first8": [float(x) for x in l32[0, :8]],
        "logits_sum": float(np.sum(l32.astype(np.float64))),
        "logprob": [float(x) for x in lp],
        "xform_idx": xidx.tolist(),
        "xform_best": [float(x) for x in xbest],
        "shard_cuts": cuts,
        "shard_idx": [s[0].tolist() for s in shards],
        "shard_logmass": [[float(x) for x in s[2]] for s in shards],
        "group_idx": gidx.tolist(),
        "group": grp.tolist(),
    }


if __name__ == "__main__":
    with open(OUT, "w") as f:
        json.dump(compute(), f, indent=1)
        f.write("\n")
    print("wrote", OUT)
