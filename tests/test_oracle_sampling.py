"""Pins for the oracle's logits and its Gumbel-max pass.

FlashSampling (arXiv 2603.15854) fixes the result as the maximizer of the
perturbed logits s_i = l~_i + g_i over the whole vocabulary (method section;
exactness by Appendix C: argmax decomposes over a partition), which is an exact
sample from softmax(l~) with l~ = l / T.  The logits are bf16 products
accumulated in f32 (the experimental setup's precision), summed in index
order.  The checks below pin the oracle to things outside itself: a
sequential float32 sum written with numpy, the textbook error bound of that
sum against an exact one, a numpy fp64 matmul for the diagnostic sums, exact
integer arithmetic, brute force on tiny vocabularies, partition invariance,
the softmax law by chi-squared tests and quadrature, and the temperature's
placement.
"""
import math

import numpy as np
import pytest
import scipy.integrate
import scipy.special
import scipy.stats
import torch

import oracle
import workloads


def bf16_bits(x):
    return workloads.to_bits(torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16))


def bits_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- logits

def sequential_f32_sum(Hf32, Wf32):
    """l[b, v] = sum_k H[b, k] W[v, k] with numpy float32: every product and
    every partial sum rounded to float32, k from 0 to D-1 (an independent
    statement of the accumulation the oracle's logits are defined by)."""
    B, D = Hf32.shape
    acc = np.zeros((B, Wf32.shape[0]), dtype=np.float32)
    for k in range(D):
        prod = (Hf32[:, k:k + 1] * Wf32[None, :, k]).astype(np.float32)
        acc = (acc + prod).astype(np.float32)
    return acc


@pytest.mark.parametrize("B,V,D", [(3, 50, 1), (2, 33, 7), (5, 129, 64), (4, 300, 257),
                                   (2, 64, 1031)])
def test_logits_equal_a_sequential_float32_sum(B, V, D):
    """Bit for bit: the oracle's logits are the f32 sum in index order.  An
    fp64 sum rounded once, another summation order (reversed, two halves) or
    a dropped term each change some of these last bits.  A fused
    multiply-add would not: a bf16 x bf16 product is exact in f32, so
    fma(h, w, acc) and acc + h * w round the same exact value."""
    rng = np.random.default_rng(B * 1000 + D)
    H = bf16_bits(rng.standard_normal((B, D)))
    W = bf16_bits(0.05 * rng.standard_normal((V, D)))
    got = oracle.logits(H, W)
    assert got.dtype == np.float32
    want = sequential_f32_sum(bits_to_f64(H).astype(np.float32), bits_to_f64(W).astype(np.float32))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("D", [64, 1000, 4096])
def test_logits_within_the_textbook_bound_of_the_exact_sum(D):
    """A recursive f32 sum of exact products errs by at most
    gamma_(D-1) * sum_k |h_k w_k|, gamma_n = n u / (1 - n u), u = 2^-24
    (Higham, Accuracy and Stability of Numerical Algorithms, recursive
    summation).  The exact sum comes from Python fractions."""
    from fractions import Fraction
    rng = np.random.default_rng(D)
    B, V = 2, 6
    H = bf16_bits(rng.standard_normal((B, D)))
    W = bf16_bits(0.02 * rng.standard_normal((V, D)))
    got = oracle.logits(H, W)
    Hf, Wf = bits_to_f64(H), bits_to_f64(W)
    u = 2.0 ** -24
    gamma = (D - 1) * u / (1 - (D - 1) * u)
    for b in range(B):
        for v in range(V):
            exact = sum(Fraction(float(Hf[b, k])) * Fraction(float(Wf[v, k])) for k in range(D))
            bound = gamma * float(np.sum(np.abs(Hf[b] * Wf[v])))
            assert abs(Fraction(float(got[b, v])) - exact) <= Fraction(bound)


@pytest.mark.parametrize("B,V,D", [(3, 50, 1), (2, 33, 7), (5, 129, 64), (4, 300, 257)])
def test_diagnostic_fp64_logits_match_numpy_matmul(B, V, D):
    rng = np.random.default_rng(B * 1000 + D)
    H = bf16_bits(rng.standard_normal((B, D)))
    W = bf16_bits(0.05 * rng.standard_normal((V, D)))
    got = oracle.logits64(H, W)
    Hf, Wf = bits_to_f64(H), bits_to_f64(W)
    want = Hf @ Wf.T
    scale = np.abs(Hf) @ np.abs(Wf).T
    assert np.all(np.abs(got - want) <= 4 * D * 2.0 ** -53 * scale + 1e-300)


def test_logits_exact_on_small_integers():
    """Small integers are exact in bf16, and every partial sum here stays an
    integer below 2^24, so both sums are the exact integers."""
    rng = np.random.default_rng(3)
    B, V, D = 3, 17, 45
    Hi = rng.integers(-8, 9, size=(B, D))
    Wi = rng.integers(-8, 9, size=(V, D))
    got = oracle.logits(bf16_bits(Hi), bf16_bits(Wi))
    got64 = oracle.logits64(bf16_bits(Hi), bf16_bits(Wi))
    for b in range(B):
        for v in range(V):
            want = sum(int(Hi[b, k]) * int(Wi[v, k]) for k in range(D))
            assert got[b, v] == want and got64[b, v] == want


def test_sample_uses_the_f32_logits():
    """oracle.sample == oracle.sample_from_logits on the oracle's f32 logits,
    and the logits it returns are those."""
    rng = np.random.default_rng(11)
    B, V, D = 6, 200, 96
    H = bf16_bits(rng.standard_normal((B, D)))
    W = bf16_bits(0.1 * rng.standard_normal((V, D)))
    T = np.array([1.0, 0.5, 1.5, 0.7, 2.0, 1.0], dtype=np.float32)
    i1, s1, t1, l32 = oracle.sample(H, W, T, 42, 9, want_logits=True)
    i2, s2, t2, _ = oracle.sample_from_logits(l32, T, 42, 9)
    assert np.array_equal(i1, i2)
    assert np.array_equal(s1, s2) and np.array_equal(t1, t2)
    assert np.array_equal(l32, oracle.logits(H, W))


# ---------------------------------------------------------------- argmax

def brute_force_row(l32, T, seed, offset, b):
    """Independent restatement on tiny V: enumerate (v, s_v) and pick the max."""
    invT = np.float32(1.0) / np.float32(T)
    pairs = []
    for v in range(len(l32)):
        g = np.float32(oracle.gumbel(seed, offset, b, v))
        s = np.float32(np.float32(l32[v]) * invT) + g
        pairs.append((float(np.float32(s)), v))
    best = max(pairs, key=lambda p: (p[0], -p[1]))
    rest = [p[0] for p in pairs if p[1] != best[1]]
    return best[1], best[0], max(rest) if rest else -math.inf


@pytest.mark.parametrize("V", [1, 2, 3, 5, 8])
def test_brute_force_tiny_vocab(V):
    rng = np.random.default_rng(V)
    B = 64
    L = rng.standard_normal((B, V)).astype(np.float32)
    T = rng.uniform(0.5, 1.5, size=B).astype(np.float32)
    idx, best, second, _ = oracle.sample_from_logits(L, T, 1234, 77)
    for b in range(B):
        i, s, s2 = brute_force_row(L[b], T[b], 1234, 77, b)
        assert idx[b] == i and best[b] == np.float32(s)
        assert second[b] == np.float32(s2)


def test_partition_invariance():
    """argmax over the whole row == max over the per-block maxima, for random
    contiguous and scattered partitions (ties resolved to the lowest index)."""
    rng = np.random.default_rng(5)
    B, V = 16, 1000
    L = rng.standard_normal((B, V)).astype(np.float32)
    L[:, 500] = L[:, 100]  # exact logit ties
    idx, best, _, S = oracle.sample_from_logits(L, 1.0, 9, 0, want_scores=True)
    for trial in range(50):
        if trial % 2 == 0:
            cuts = np.sort(rng.choice(np.arange(1, V), size=rng.integers(1, 40), replace=False))
            blocks = np.split(np.arange(V), cuts)
        else:
            perm = rng.permutation(V)
            blocks = np.array_split(perm, rng.integers(2, 30))
        for b in range(B):
            cands = []
            for blk in blocks:
                blk = np.sort(blk)
                j = blk[np.argmax(S[b, blk])]  # np.argmax: first occurrence
                cands.append((S[b, j], -j))
            s, negj = max(cands)
            assert -negj == idx[b] and s == best[b]


def test_ties_go_to_lowest_index_without_noise():
    L = np.zeros((4, 64), dtype=np.float32)
    L[0, [5, 9, 40]] = 3.0
    L[1, :] = 1.0
    L[2, [63, 62]] = 2.0
    L[3, [0, 63]] = -1.0
    L[3, 1:63] = -2.0
    idx, best, second, _ = oracle.sample_from_logits(L, 1.0, 0, 0, flags=oracle.NO_NOISE)
    assert list(idx) == [5, 0, 62, 0]
    assert list(best) == [3.0, 1.0, 2.0, -1.0]
    assert list(second) == [3.0, 1.0, 2.0, -1.0]  # equal runner-up => gap 0


def test_invalid_temperature_and_nonfinite_logits():
    L = np.ones((6, 16), dtype=np.float32)
    T = np.array([0.0, -1.0, np.inf, np.nan, 1.0, 1.0], dtype=np.float32)
    L[4, :] = np.nan
    L[5, :] = -np.inf
    L[5, 7] = 0.0
    idx, best, second, _ = oracle.sample_from_logits(L, T, 3, 0)
    assert list(idx[:4]) == [-1, -1, -1, -1]
    assert np.all(np.isnan(best[:4])) and np.all(np.isnan(second[:4]))
    assert idx[4] == -1 and best[4] == -np.inf  # NaN never wins
    assert idx[5] == 7  # the only finite score wins


def test_temperature_divides_logits_before_the_noise():
    """T = 2 is exact in f32: sample(l, T=2) == sample(l/2, T=1) bit for bit,
    and differs from argmax(l + g) (noise added before the division)."""
    rng = np.random.default_rng(8)
    L = (3 * rng.standard_normal((4096, 16))).astype(np.float32)
    a = oracle.sample_from_logits(L, 2.0, 21, 4)[0]
    b = oracle.sample_from_logits(L / np.float32(2.0), 1.0, 21, 4)[0]
    c = oracle.sample_from_logits(L, 1.0, 21, 4)[0]
    assert np.array_equal(a, b)
    assert np.count_nonzero(a != c) > 100


# ---------------------------------------------------------------- distribution

def chisq_pvalue(counts, probs):
    n = counts.sum()
    exp = probs * n
    # merge categories with expected count < 5 into one bucket
    small = exp < 5
    if small.any():
        counts = np.append(counts[~small], counts[small].sum())
        exp = np.append(exp[~small], exp[small].sum())
        if exp[-1] == 0:
            counts, exp = counts[:-1], exp[:-1]
    return scipy.stats.chisquare(counts, exp).pvalue


def softmax_f32_transform(l, T):
    invT = np.float32(1.0) / np.float32(T)
    lt = (l.astype(np.float32) * invT).astype(np.float64)
    return scipy.special.softmax(lt)


@pytest.mark.parametrize("V", [2, 8, 64])
@pytest.mark.parametrize("T", [0.5, 1.0, 1.5])
def test_frequencies_match_softmax_across_rows(V, T):
    """10^5 draws (one per row, distinct Philox counters) vs softmax(l/T)."""
    rng = np.random.default_rng(100 * V + int(10 * T))
    l = (1.5 * rng.standard_normal(V)).astype(np.float32)
    N = 100_000
    L = np.broadcast_to(l, (N, V))
    idx = oracle.sample_from_logits(L, T, 0xC0FFEE + V, 0)[0]
    counts = np.bincount(idx, minlength=V).astype(np.float64)
    assert chisq_pvalue(counts, softmax_f32_transform(l, T)) > 0.01


def test_frequencies_match_softmax_across_offsets():
    """10^5 decode steps (offset = step) of one row vs softmax(l/T)."""
    V, T, N = 8, 0.8, 100_000
    l = np.array([0.3, -1.0, 2.0, 0.0, 1.1, -0.4, 0.9, 2.0], dtype=np.float32)
    counts = np.zeros(V)
    for off in range(N):
        counts[oracle.sample_from_logits(l[None, :], T, 0xABCD, off)[0][0]] += 1
    assert chisq_pvalue(counts, softmax_f32_transform(l, T)) > 0.01


def test_duplicates_sampled_with_equal_frequency():
    V, N = 16, 100_000
    l = np.linspace(-1, 1, V).astype(np.float32)
    l[9] = l[3]
    l[15] = l[3]
    idx = oracle.sample_from_logits(np.broadcast_to(l, (N, V)), 1.0, 0xD00D, 0)[0]
    c = np.bincount(idx, minlength=V)
    trio = np.array([c[3], c[9], c[15]], dtype=np.float64)
    assert scipy.stats.chisquare(trio).pvalue > 0.01


def test_gumbel_max_law_by_quadrature():
    """P(i wins) = int pdf(x - l_i) prod_{j != i} F(x - l_j) dx equals
    softmax(l)_i: the law the chi-squared tests compare against."""
    l = np.array([0.5, -1.0, 2.0, 0.1])
    pdf = lambda x: np.exp(-x - np.exp(-x))
    cdf = lambda x: np.exp(-np.exp(-x))
    for i in range(len(l)):
        f = lambda x: pdf(x - l[i]) * np.prod([cdf(x - l[j]) for j in range(len(l)) if j != i])
        p, _ = scipy.integrate.quad(f, -20, 40, limit=200)
        assert abs(p - scipy.special.softmax(l)[i]) < 1e-8


def test_row_ids_key_the_noise_like_the_full_batch():
    """Sampling a subset of rows with their batch indices reproduces the
    full-batch result for those rows (used for sampled-row parity checks)."""
    rng = np.random.default_rng(12)
    B, V, D = 9, 70, 24
    H = bf16_bits(rng.standard_normal((B, D)))
    W = bf16_bits(0.2 * rng.standard_normal((V, D)))
    T = rng.uniform(0.5, 1.5, size=B).astype(np.float32)
    full = oracle.sample(H, W, T, 5, 6)
    rows = np.array([7, 2, 8])
    sub = oracle.sample(H[rows], W, T[rows], 5, 6, row_ids=rows)
    for a, b in zip(full[:3], sub[:3]):
        assert np.array_equal(a[rows], b)


# ---------------------------------------------------------------- log-probability

def test_logprob_matches_scipy_log_softmax():
    """The sampled token's log-probability (the log-mass summary) against
    scipy's log_softmax of the same f32-transformed logits."""
    rng = np.random.default_rng(31)
    B, V = 7, 5000
    L = (2.5 * rng.standard_normal((B, V))).astype(np.float32)
    T = rng.uniform(0.3, 2.0, size=B).astype(np.float32)
    idx = oracle.sample_from_logits(L, T, 3, 4)[0]
    got = oracle.logprob(L, T, idx)
    for b in range(B):
        lt = (L[b] * (np.float32(1.0) / T[b])).astype(np.float64)
        want = scipy.special.log_softmax(lt)[idx[b]]
        assert abs(got[b] - want) < 1e-10


def test_logprob_closed_forms():
    V = 1000
    L = np.zeros((3, V), dtype=np.float32)
    L[1, 7] = 50.0  # one dominant token
    L[2, :] = np.float32(-1e30)  # huge negative but equal
    idx = np.array([5, 7, 999])
    got = oracle.logprob(L, np.ones(3, dtype=np.float32), idx)
    assert abs(got[0] - (-np.log(V))) < 1e-12
    assert abs(got[1] - (-np.log1p((V - 1) * np.exp(-50.0)))) < 1e-12
    assert abs(got[2] - (-np.log(V))) < 1e-12
    bad = oracle.logprob(L, np.array([1.0, 0.0, 1.0], dtype=np.float32), np.array([-1, 3, 2]))
    assert np.isnan(bad[0]) and np.isnan(bad[1]) and not np.isnan(bad[2])


def test_logprob_probabilities_sum_to_one():
    rng = np.random.default_rng(2)
    V = 300
    l = (3 * rng.standard_normal(V)).astype(np.float32)
    L = np.broadcast_to(l, (V, V))
    lp = oracle.logprob(L, np.full(V, 0.7, dtype=np.float32), np.arange(V))
    assert abs(np.exp(lp).sum() - 1.0) < 1e-12


def test_logprob_leaves_out_non_finite_logits():
    """Reading for non-finite l~ (the pages are silent): the log-mass runs over
    the finite entries; a sampled token with a non-finite l~ gets NaN."""
    l = np.array([0.5, -np.inf, 1.0, np.nan, -0.25, np.inf], dtype=np.float32)
    L = np.broadcast_to(l, (3, 6))
    got = oracle.logprob(L, np.ones(3, dtype=np.float32), np.array([0, 2, 5]))
    finite = np.array([0.5, 1.0, -0.25])
    ref = scipy.special.log_softmax(finite)
    assert abs(got[0] - ref[0]) < 1e-12 and abs(got[1] - ref[1]) < 1e-12
    assert np.isnan(got[2])


# ---------------------------------------------------------------- deterministic transforms

def test_transforms_bias_softcap_mask():
    """Bias, soft-capping and the allowed-token mask, checked elementwise
    against numpy float32 arithmetic and bit tests."""
    rng = np.random.default_rng(41)
    B, V = 3, 100
    L = (8 * rng.standard_normal((B, V))).astype(np.float32)
    bias = rng.standard_normal(V).astype(np.float32)
    words = 4
    mask = rng.integers(0, 2**32, size=(B, words), dtype=np.uint64).astype(np.uint32)
    out = oracle.transform_logits(L, bias, 30.0, mask)
    want = (L + bias).astype(np.float32)
    want = (np.float32(30.0) * np.tanh(want / np.float32(30.0))).astype(np.float32)
    allowed = np.array([[(int(mask[b, v // 32]) >> (v % 32)) & 1 for v in range(V)]
                        for b in range(B)], dtype=bool)
    assert np.all(out[~allowed] == -np.inf)
    assert np.allclose(out[allowed], want[allowed], rtol=2e-7, atol=0)
    assert np.all(np.abs(out[allowed]) < 30.0)
    # identity when nothing is set
    assert np.array_equal(oracle.transform_logits(L), L)


def test_masked_tokens_are_never_sampled():
    rng = np.random.default_rng(43)
    B, V = 2000, 40
    L = np.broadcast_to(rng.standard_normal(V).astype(np.float32), (B, V))
    mask = np.zeros((B, 2), dtype=np.uint32)
    mask[:, 0] = 0b1010_0000_0000_0000_0000_0000_0001_0110  # tokens 1, 2, 4, 29, 31
    mask[:, 1] = 1 << 3                                     # token 35
    out = oracle.transform_logits(L, mask=mask)
    idx = oracle.sample_from_logits(out, 1.0, 5, 0)[0]
    assert set(np.unique(idx)) <= {1, 2, 4, 29, 31, 35}
    counts = np.bincount(idx, minlength=V)[[1, 2, 4, 29, 31, 35]].astype(np.float64)
    p = scipy.special.softmax(l[[1, 2, 4, 29, 31, 35]].astype(np.float64)) if (l := L[0]) is not None else None
    assert scipy.stats.chisquare(counts, p * B).pvalue > 0.01


# ---------------------------------------------------------------- grouped (hierarchical) sampling

def _shard_bounds(V, cuts):
    b = [0] + list(cuts) + [V]
    return list(zip(b[:-1], b[1:]))


def test_one_group_is_the_plain_sample():
    """With a single group the grouped sampler returns the plain Gumbel-max
    sample; a shard's local sample is the global pass restricted to it."""
    rng = np.random.default_rng(51)
    B, V, D = 6, 96, 24
    H = bf16_bits(rng.standard_normal((B, D)))
    W = bf16_bits(0.3 * rng.standard_normal((V, D)))
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    idx_full = oracle.sample(H, W, T, 8, 2)[0]
    i1, s1, lm1, _ = oracle.sample_shard(H, W, 0, T, 8, 2)
    assert np.array_equal(i1, idx_full)
    out, grp = oracle.combine_groups(i1[None, :], lm1[None, :], 8, 2)
    assert np.array_equal(out, idx_full) and np.all(grp == 0)
    # a shard's log-mass is scipy's logsumexp of its l~
    l32 = oracle.logits(H, W)
    i2, s2, lm2, _ = oracle.sample_shard(H, W[32:80], 32, T, 8, 2)
    for b in range(B):
        lt = (l32[b, 32:80] * (np.float32(1) / T[b])).astype(np.float64)
        assert abs(lm2[b] - scipy.special.logsumexp(lt)) < 1e-10
        full_scores = oracle.sample_from_logits(l32[b:b + 1], T[b], 8, 2, want_scores=True,
                                                row_ids=[b])[3][0]
        assert i2[b] == 32 + int(np.argmax(full_scores[32:80]))


def test_group_noise_is_separate_from_token_noise():
    a = np.array([oracle.group_gumbel(5, 1, 3, g) for g in range(64)])
    b = np.array([oracle.gumbel(5, 1, 3, g) for g in range(64)])
    assert np.count_nonzero(a == b) == 0


def _tied_logmass(seed, offset, b, g_lo, g_hi):
    """A log-mass for group g_hi whose f32 sum with its Gumbel equals group
    g_lo's sum at log-mass 0, searched over a few floats around the
    difference of the two Gumbels."""
    G = [np.float32(oracle.group_gumbel(seed, offset, b, g)) for g in (g_lo, g_hi)]
    target = np.float32(np.float32(0) + G[0])
    x = np.float32(G[0] - G[1])
    for k in range(-8, 9):
        cand = np.float32(x + np.float32(k) * np.spacing(x))
        if np.float32(cand + G[1]) == target:
            return cand
    raise AssertionError("no exact tie found")


def test_group_ties_go_to_the_lower_group():
    """Ties between groups' perturbed log-masses go to the lower group (the
    same rule as for tokens); NaN and -inf log-masses never win."""
    seed, offset = 12, 3
    # row 0: groups 0 and 1 tie; row 1: groups 1 and 2 tie, group 0 is -inf
    t01 = _tied_logmass(seed, offset, 0, 0, 1)
    t12 = _tied_logmass(seed, offset, 1, 1, 2)
    lm = np.array([[0.0, -np.inf], [t01, 0.0], [-np.inf, t12]], dtype=np.float32)
    idx = np.array([[10, 20], [11, 21], [12, 22]], dtype=np.int64)
    out, grp, best, second = oracle.combine_groups(idx, lm, seed, offset, want_scores=True)
    assert best[0] == second[0] and best[1] == second[1]  # the ties are exact
    assert list(grp) == [0, 1] and list(out) == [10, 21]
    # NaN never wins, even against -inf; a row of only -inf / NaN has no group
    lm2 = np.array([[np.nan, np.nan], [-np.inf, np.nan]], dtype=np.float32)
    out2, grp2 = oracle.combine_groups(idx[:2], lm2, seed, offset)
    assert list(grp2) == [-1, -1] and list(out2) == [-1, -1]


@pytest.mark.parametrize("cuts", [(16,), (8, 40), (3, 5, 30, 31)])
def test_grouped_sampler_matches_softmax(cuts):
    """Hierarchical factorisation: 10^5 grouped draws (rows as trials) follow
    softmax(l/T) whatever the grouping.  Each group's local sample is the
    Gumbel-max over the group with the noise of the global indices; its
    log-mass is scipy's logsumexp of the group's l~."""
    rng = np.random.default_rng(sum(cuts))
    V, N, T = 48, 100_000, 0.9
    l = (1.3 * rng.standard_normal(V)).astype(np.float32)
    invT = np.float32(1) / np.float32(T)
    gidx, glm = [], []
    for v0, v1 in _shard_bounds(V, cuts):
        _, g = oracle.noise_block(77, 0, 0, N, v0, v1 - v0)
        lt = (l[v0:v1] * invT).astype(np.float32)
        gidx.append(v0 + np.argmax((lt[None, :] + g).astype(np.float32), axis=1))
        glm.append(np.full(N, scipy.special.logsumexp(lt.astype(np.float64))))
    out, grp = oracle.combine_groups(np.stack(gidx), np.stack(glm), 91, 0)
    counts = np.bincount(out, minlength=V).astype(np.float64)
    assert chisq_pvalue(counts, softmax_f32_transform(l, T)) > 0.01
