"""The inequality behind Stage 1's per-element screen, checked exhaustively.

The screen rejects an element when 2^-23 * e2 >= exp(lt - best), with
e2 = (~x) >> 9 taken from the element's 32-bit random word x.  That is safe
only if 2^-23 * e2 never exceeds w = -log(u), u = ((x >> 8) | 1) * 2^-24, so
that a rejected element's Gumbel -log(w) is at most best - lt.  u and e2
depend on x only through x >> 8, so all 2^24 values are checked.
"""
import numpy as np


def test_tail_bound_never_exceeds_minus_log_u():
    a = np.arange(1 << 24, dtype=np.uint64)           # x >> 8
    u = (a | 1).astype(np.float64) * 2.0 ** -24
    x = (a << 8).astype(np.uint32)                     # any low byte gives the same e2
    e2 = ((~x) >> 9).astype(np.float64)
    assert np.array_equal(e2, ((0xFFFFFF - a) >> 1).astype(np.float64))
    w = -np.log(u)
    assert np.all(e2 * 2.0 ** -23 <= w)
    # and it is tight where the screen decides (u near 1): within a factor 2/3
    near = (u > 0.999) & (e2 > 0)
    assert np.min(e2[near] * 2.0 ** -23 / w[near]) > 0.66
