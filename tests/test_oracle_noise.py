"""Pins for the oracle's noise: Philox4x64-10, the uniform map and the Gumbel.

The oracle's generator is checked against numpy's own Philox4x64-10 bit
generator (an independent library implementation of the SC'11 definition),
the uniform map exhaustively over its whole 2^24-value domain, and the Gumbel
transform through its inverse (the Gumbel CDF), its closed-form moments and a
KS test.  FlashSampling draws "i.i.d. Gumbels" (method section); the generator
itself is this library's reading (the pages name none).
"""
import math

import numpy as np
import pytest
import scipy.stats

import oracle

MASK64 = (1 << 64) - 1


def numpy_block(counter_words, key_words):
    """Philox4x64-10 block at `counter` computed by numpy's bit generator.

    numpy increments its 256-bit counter before producing a block, so the
    block at counter c is the first output of a generator set to c - 1.
    """
    c = sum(int(w) << (64 * i) for i, w in enumerate(counter_words))
    k = int(key_words[0]) | (int(key_words[1]) << 64)
    bg = np.random.Philox(counter=(c - 1) % (1 << 256), key=k)
    return [int(x) for x in bg.random_raw(4)]


def test_philox_matches_numpy_random_counters():
    rng = np.random.default_rng(12345)
    for _ in range(2000):
        ctr = [int(x) for x in rng.integers(0, 2**64, size=4, dtype=np.uint64)]
        key = [int(x) for x in rng.integers(0, 2**64, size=2, dtype=np.uint64)]
        got = [int(x) for x in oracle.philox4x64_10(ctr, key)]
        assert got == numpy_block(ctr, key), (ctr, key)


@pytest.mark.parametrize("ctr,key", [
    ([0, 0, 0, 0], [0, 0]),
    ([1, 0, 0, 0], [0, 0]),
    ([MASK64, MASK64, MASK64, MASK64], [MASK64, MASK64]),
    ([0, 1, 0, 0], [0x5EED0040, 0]),
    ([16031, 63, 7, 0], [0x5EED0040, 0]),
    ([MASK64, 0, 0, 0], [1, 2]),
])
def test_philox_matches_numpy_edge_counters(ctr, key):
    got = [int(x) for x in oracle.philox4x64_10(ctr, key)]
    assert got == numpy_block(ctr, key)


def test_noise_word_layout_matches_numpy():
    """Element (b, v) draws half (v & 1) of word (v & 7) >> 1 of the block at
    counter (v >> 3, b, offset, 0) under key (seed, 0)."""
    rng = np.random.default_rng(7)
    for _ in range(300):
        seed = int(rng.integers(0, 2**64, dtype=np.uint64))
        offset = int(rng.integers(0, 2**64, dtype=np.uint64))
        b = int(rng.integers(0, 1 << 20))
        v = int(rng.integers(0, 1 << 31))
        blk = numpy_block([v >> 3, b, offset, 0], [seed, 0])
        w = blk[(v & 7) >> 1]
        want = (w >> 32) if (v & 1) else (w & 0xFFFFFFFF)
        assert oracle.noise_word(seed, offset, b, v) == want


def test_noise_block_equals_pointwise():
    words, g = oracle.noise_block(99, 5, 3, 4, 17, 37)
    for i in range(4):
        for j in range(37):
            assert words[i, j] == oracle.noise_word(99, 5, 3 + i, 17 + j)
            assert g[i, j] == np.float32(oracle.gumbel(99, 5, 3 + i, 17 + j))


def test_uniform_exhaustive():
    """All 2^24 values of x >> 8: u is exact, in (0, 1), symmetric, uniform."""
    k = np.arange(1 << 24, dtype=np.uint64)
    x = (k << np.uint64(8)).astype(np.uint32)
    u = oracle.uniform_block(x)
    assert np.all(u > 0.0) and np.all(u < 1.0)
    # low 8 bits never matter
    assert np.array_equal(oracle.uniform_block(x | np.uint32(0xFF)), u)
    # every u is an odd multiple of 2^-24 and each odd numerator appears twice
    num = u * (1 << 24)
    assert np.array_equal(num, np.floor(num))
    numi = num.astype(np.int64)
    assert np.all(numi % 2 == 1)
    counts = np.bincount(numi, minlength=1 << 24)
    assert np.all(counts[1::2] == 2) and np.all(counts[0::2] == 0)
    # symmetric: u(k) + u(2^24 - 1 - k) = 1, hence mean exactly 1/2
    assert np.array_equal(u + u[::-1], np.ones_like(u))
    assert u.sum() == (1 << 23)
    assert u.min() == 2.0 ** -24 and u.max() == 1.0 - 2.0 ** -24


def test_gumbel_inverts_the_gumbel_cdf():
    """F(g) = exp(-exp(-g)) must give back u up to the f32 rounding of g.

    |F(g32) - u| <= max|F'| * |g32 - g| <= (1/e) * ulp(g)/2 (+ fp64 noise)."""
    k = np.arange(0, 1 << 24, 97, dtype=np.uint64)
    k = np.concatenate([k, np.arange(0, 4096, dtype=np.uint64),
                        np.arange((1 << 24) - 4096, 1 << 24, dtype=np.uint64)])
    x = (k << np.uint64(8)).astype(np.uint32)
    u = oracle.uniform_block(x)
    g = oracle.gumbel_block(x).astype(np.float64)
    F = np.exp(-np.exp(-g))
    ulp = np.spacing(np.abs(g).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(F - u) <= 0.19 * ulp + 1e-15)
    # monotone in u, and the extreme values sit where the closed form says
    order = np.argsort(u, kind="stable")
    assert np.all(np.diff(g[order]) >= 0)
    assert abs(g.max() - (-math.log(-math.log1p(-2.0 ** -24)))) < 1e-5
    assert abs(g.min() - (-math.log(24 * math.log(2.0)))) < 1e-5


def test_gumbel_moments_and_ks():
    """Mean = Euler-Mascheroni constant, variance = pi^2/6, KS vs the Gumbel CDF."""
    _, g = oracle.noise_block(0x1234, 0, 0, 64, 0, 1 << 14)
    g = g.ravel().astype(np.float64)
    n = g.size
    se_mean = math.sqrt(math.pi ** 2 / 6 / n)
    assert abs(g.mean() - 0.5772156649015329) < 5 * se_mean
    # var of the sample variance of a Gumbel: (mu4 - sigma^4)/n, mu4 = 5.4 sigma^4
    s2 = math.pi ** 2 / 6
    se_var = math.sqrt((5.4 - 1.0) * s2 * s2 / n)
    assert abs(g.var() - s2) < 5 * se_var
    p = scipy.stats.kstest(g, scipy.stats.gumbel_r.cdf).pvalue
    assert p > 0.01


def test_noise_words_bits_balanced_across_layout():
    """Each of the 32 bits is set half the time, separately for even/odd v and
    for each of the four 64-bit words: catches a layout that reuses a half."""
    words, _ = oracle.noise_block(77, 3, 0, 32, 0, 8192)
    w = words.reshape(32, 1024, 8)
    for j in range(8):
        lane = w[:, :, j].ravel().astype(np.uint64)
        n = lane.size
        for bit in range(32):
            ones = int(((lane >> np.uint64(bit)) & np.uint64(1)).sum())
            assert abs(ones - n / 2) < 5 * math.sqrt(n / 4), (j, bit)
    # neighbouring elements are not equal more often than chance (2^-32)
    flat = words.ravel()
    assert np.count_nonzero(flat[1:] == flat[:-1]) <= 2


def test_offsets_and_rows_give_independent_streams():
    a, _ = oracle.noise_block(5, 0, 0, 1, 0, 4096)
    b, _ = oracle.noise_block(5, 1, 0, 1, 0, 4096)
    c, _ = oracle.noise_block(5, 0, 1, 1, 0, 4096)
    d, _ = oracle.noise_block(6, 0, 0, 1, 0, 4096)
    for other in (b, c, d):
        assert np.count_nonzero(a == other) <= 2


def test_largest_gumbel_is_the_closed_form_at_the_largest_uniform():
    """The largest uniform is u = 1 - 2^-24, so no Gumbel exceeds
    -log(-log(1 - 2^-24)) = 16.6355...; over all 2^23 distinct uniforms the
    oracle's largest Gumbel is that closed form, reached at the last one."""
    k = np.arange(1, 1 << 24, 2, dtype=np.uint32)
    g = oracle.gumbel_block(k << np.uint32(8))
    g_max = -math.log(-math.log1p(-2.0 ** -24))
    assert abs(float(g.max()) - g_max) < 1e-5
    assert int(np.argmax(g)) == len(k) - 1  # at u = 1 - 2^-24
