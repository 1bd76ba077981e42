"""Seeded synthetic inputs for the LM-head + sampling workloads.

This module only draws random inputs; it holds none of the sampling method's
arithmetic.  Both the CUDA path and the CPU oracle are fed from here: tests
generate a tensor once and hand the oracle a host copy of exactly those bits.

The workloads stand in for the LM heads the FlashSampling pages measure
(decode configuration D=4096/V=151936 and the larger D=8192/V=128256 one of
the experimental setup and tensor-parallel sections).  No trained weights are
used; only the shapes, dtypes (bf16, as the pages state for inputs and
weights) and value distributions below are taken.

Recipes (sigma is a standard deviation):
  tiny       D=256,  V=4096;   H ~ N(0,1); W ~ N(0, 1/sqrt(D)); T = 1.0
  llama3_8b  D=4096, V=128256; H ~ N(0,1), each row scaled to RMS 1;
             W ~ N(0, 0.02); T = 1.0
  qwen       D=3584, V=151936; H ~ N(0,1) with column D-1 set to 1;
             W ~ N(0, 0.02) with column D-1 holding a Zipf-like bias
             -alpha * ln(rank_v) (rank = seeded permutation of 1..V,
             alpha = 2.75 so the logit std is about 3); per-row T ~ U[0.5, 1.5]
  llama3_70b D=8192, V=128256; H ~ N(0,1); W ~ N(0, 0.015); T = 0.7
  bigvocab   D=2304, V=262144; H ~ N(0,1); W ~ N(0, 0.02); 1% of the rows
             (seeded pick, never row 0) are exact copies of a lower-index row,
             which forces exact logit ties; T = 1.0

Every generator accepts V/D overrides so that the CPU tests can use the same
recipe at small sizes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

__all__ = ["Workload", "WORKLOADS", "make_weights", "make_hidden",
           "make_temperature", "sampling_seed", "to_bits"]


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    D: int
    V: int
    batches: tuple
    w_sigma: float
    temperature: float | None  # None -> per-row U[0.5, 1.5]


WORKLOADS = {
    "tiny": Workload("tiny", 0, 256, 4096, (4,), 1.0 / 16.0, 1.0),
    "llama3_8b": Workload("llama3_8b", 1, 4096, 128256, (1, 2, 4, 8, 16, 32, 64), 0.02, 1.0),
    "qwen": Workload("qwen", 2, 3584, 151936, (1, 2, 4, 8, 16, 32, 64, 128, 256), 0.02, None),
    "llama3_70b": Workload("llama3_70b", 3, 8192, 128256, (256, 512, 1024), 0.015, 0.7),
    "bigvocab": Workload("bigvocab", 4, 2304, 262144, (1, 8, 64, 512), 0.02, 1.0),
}

QWEN_BIAS_ALPHA = 2.75
DUP_FRACTION = 0.01


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_weights(name: str, device="cpu", V: int | None = None, D: int | None = None,
                 seed: int | None = None) -> torch.Tensor:
    """LM-head weight W [V, D] bf16, row-major (vocab-major)."""
    wl = WORKLOADS[name]
    V = wl.V if V is None else int(V)
    D = wl.D if D is None else int(D)
    seed = 1000 + wl.index if seed is None else seed
    g = _gen(device, seed)
    W = torch.empty((V, D), dtype=torch.bfloat16, device=device)
    chunk = max(1, (1 << 26) // max(D, 1))
    for r0 in range(0, V, chunk):
        r1 = min(V, r0 + chunk)
        x = torch.randn((r1 - r0, D), generator=g, device=device, dtype=torch.float32)
        W[r0:r1] = (x * wl.w_sigma).to(torch.bfloat16)
    if name == "qwen":
        rank = torch.randperm(V, generator=g, device=device).to(torch.float64) + 1.0
        W[:, D - 1] = (-QWEN_BIAS_ALPHA * torch.log(rank)).to(torch.bfloat16)
    if name == "bigvocab" and V > 1:
        n_dup = max(1, int(V * DUP_FRACTION))
        n_dup = min(n_dup, V - 1)
        targets = torch.randperm(V - 1, generator=g, device=device)[:n_dup] + 1
        u = torch.rand(n_dup, generator=g, device=device, dtype=torch.float64)
        src = torch.clamp((u * targets.to(torch.float64)).floor().to(torch.int64),
                          max=targets - 1)
        # Follow copy chains down to a row that is not itself overwritten, so
        # every copied row ends equal to an untouched lower-index row.
        src_of = torch.arange(V, device=device)
        src_of[targets] = src
        is_target = torch.zeros(V, dtype=torch.bool, device=device)
        is_target[targets] = True
        root = src.clone()
        for _ in range(64):
            nxt = torch.where(is_target[root], src_of[root], root)
            if torch.equal(nxt, root):
                break
            root = nxt
        W[targets] = W[root]
    return W


def make_hidden(name: str, B: int, device="cpu", D: int | None = None,
                seed: int | None = None) -> torch.Tensor:
    """Hidden states H [B, D] bf16, row-major."""
    wl = WORKLOADS[name]
    D = wl.D if D is None else int(D)
    seed = 2000 + wl.index * 4096 + B if seed is None else seed
    g = _gen(device, seed)
    x = torch.randn((B, D), generator=g, device=device, dtype=torch.float32)
    if name == "llama3_8b":
        x = x / torch.sqrt(torch.mean(x * x, dim=1, keepdim=True))
    if name == "qwen" and D > 0:
        x[:, D - 1] = 1.0
    return x.to(torch.bfloat16)


def make_temperature(name: str, B: int, device="cpu", seed: int | None = None):
    """Scalar float, or a per-row f32 tensor [B] for the per-row workloads."""
    wl = WORKLOADS[name]
    if wl.temperature is not None:
        return float(wl.temperature)
    seed = 3000 + wl.index * 4096 + B if seed is None else seed
    g = _gen(device, seed)
    return (0.5 + torch.rand(B, generator=g, device=device, dtype=torch.float32)).contiguous()


def sampling_seed(name: str, B: int):
    """(seed, offset) of the sampling call for a workload and batch size."""
    return 0x5EED0000 + int(B), 0


def to_bits(t: torch.Tensor):
    """Raw uint16 words of a bf16 tensor as a host numpy array."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def logit_std_estimate(name: str) -> float:
    """Approximate standard deviation of the logits of a workload's recipe."""
    wl = WORKLOADS[name]
    base = wl.w_sigma * math.sqrt(wl.D)
    if name == "qwen":
        return math.sqrt(wl.w_sigma ** 2 * (wl.D - 1) + QWEN_BIAS_ALPHA ** 2)
    return base
