"""The seeded synthetic inputs follow their stated recipes (workloads/synth.py).

Checked at reduced V / D, which the generators accept, so the CPU suite stays
fast: shapes and dtypes, determinism, the per-workload structure (RMS-scaled
rows, the Zipf-like bias column, exact duplicate rows, per-row temperatures).
"""
import numpy as np
import torch

import workloads


def test_shapes_dtypes_and_determinism():
    for name, wl in workloads.WORKLOADS.items():
        W = workloads.make_weights(name, V=1000, D=64)
        H = workloads.make_hidden(name, 5, D=64)
        assert W.shape == (1000, 64) and W.dtype == torch.bfloat16 and W.is_contiguous()
        assert H.shape == (5, 64) and H.dtype == torch.bfloat16
        assert torch.equal(W, workloads.make_weights(name, V=1000, D=64))
        assert torch.equal(H, workloads.make_hidden(name, 5, D=64))
        assert not torch.equal(H, workloads.make_hidden(name, 6, D=64)[:5])  # seed keyed by B


def test_weight_scale_matches_the_recipe():
    W = workloads.make_weights("llama3_8b", V=4000, D=256).float()
    assert abs(W.std().item() - 0.02) < 0.001
    W = workloads.make_weights("llama3_70b", V=4000, D=256).float()
    assert abs(W.std().item() - 0.015) < 0.001


def test_llama3_8b_rows_have_unit_rms():
    H = workloads.make_hidden("llama3_8b", 16, D=512).float()
    rms = H.pow(2).mean(dim=1).sqrt()
    assert torch.all((rms - 1).abs() < 0.01)  # bf16 rounding only


def test_qwen_bias_column_is_minus_alpha_log_rank():
    V, D = 3000, 32
    W = workloads.make_weights("qwen", V=V, D=D)
    H = workloads.make_hidden("qwen", 4, D=D)
    assert torch.all(H[:, D - 1].float() == 1.0)
    bias = W[:, D - 1].float().numpy()
    expect = (-workloads.synth.QWEN_BIAS_ALPHA * np.log(np.arange(1, V + 1))).astype(np.float32)
    expect = torch.tensor(expect).to(torch.bfloat16).float().numpy()
    assert np.array_equal(np.sort(bias), np.sort(expect))  # a permutation of the ranks
    assert bias.max() == 0.0 and not np.array_equal(bias, expect)  # shuffled


def test_bigvocab_duplicates_are_exact_copies_of_lower_rows():
    V, D = 5000, 16
    W = workloads.make_weights("bigvocab", V=V, D=D)
    Wn = W.view(torch.int16).numpy()
    _, first, inverse = np.unique(Wn, axis=0, return_index=True, return_inverse=True)
    inverse = inverse.reshape(-1)
    is_copy = first[inverse] != np.arange(V)
    n = int(is_copy.sum())
    assert n == int(V * workloads.synth.DUP_FRACTION)  # every planted copy, nothing else
    assert not is_copy[0]
    assert np.all(first[inverse][is_copy] < np.nonzero(is_copy)[0])


def test_temperatures():
    assert workloads.make_temperature("llama3_8b", 8) == 1.0
    assert workloads.make_temperature("llama3_70b", 8) == 0.7
    T = workloads.make_temperature("qwen", 1000)
    assert T.shape == (1000,) and T.dtype == torch.float32
    assert float(T.min()) >= 0.5 and float(T.max()) < 1.5
    assert abs(float(T.mean()) - 1.0) < 0.05
