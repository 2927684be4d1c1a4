"""The range over which a compensated fp32 square is exact, as the CUDA kernels form it for their
norms: p = fl32(c*c) and e = fl32(c*c - p) (one FMA), so that p + e = c*c.  The residual c*c - p
needs the bits of c*c below p's last place, which land on fp32's subnormal grid once c is small.
The claim checked here: p + e equals c*c exactly for every fp32 |c| >= 2^-51, and not for every c
below that.  No GPU needed: an FMA's result is the correctly rounded c*c - p, which double
arithmetic gives exactly here (c*c and p are exact in double)."""
import numpy as np


def _pair(c):
    c64 = c.astype(np.float64)
    p = (c * c).astype(np.float32)                       # fp32 product, correctly rounded
    e = (c64 * c64 - p.astype(np.float64)).astype(np.float32)  # the FMA residual, rounded once
    return p, e


def _exact(c):
    p, e = _pair(c)
    c64 = c.astype(np.float64)
    return p.astype(np.float64) + e.astype(np.float64) == c64 * c64


def test_squares_are_exact_down_to_two_to_the_minus_51():
    rng = np.random.default_rng(0)
    for k in range(-51, 63):  # every binade from 2^-51 up to just below 2^64 (c*c below FLT_MAX)
        m = rng.integers(1 << 23, 1 << 24, size=4096).astype(np.float64)
        c = np.ldexp(m, k - 23).astype(np.float32)  # full 24-bit significands in [2^k, 2^(k+1))
        assert np.all(_exact(c)), k


def test_squares_lose_exactness_below_that():
    rng = np.random.default_rng(1)
    for k in (-52, -55, -60, -63):
        m = rng.integers(1 << 23, 1 << 24, size=4096).astype(np.float64)
        c = np.ldexp(m, k - 23).astype(np.float32)
        assert not np.all(_exact(c)), k
    # far below, the square itself is gone
    tiny = np.float32(2.0 ** -76)
    p, e = _pair(np.array([tiny]))
    assert p[0] == 0 and e[0] == 0
