"""The range over which a compensated fp32 square is exact, as the CUDA kernels form it for their
norms: p = fl32(c*c) and e = fl32(c*c - p) (one FMA), so that p + e = c*c.  The residual c*c - p
needs the bits of c*c below p's last place, which land on fp32's subnormal grid once c is small.
The claim checked here: p + e equals c*c exactly for every fp32 |c| >= 2^-51, and not for every c
below that; and the unit-level range check that sends every unit outside [2^-56, 2^100) to a
double-precision sum (below).  No GPU needed: an FMA's result is the correctly rounded c*c - p, which double
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


# ---- the unit-level range check of the kernels' norms
#
# The kernels accumulate each thread's squares as fp32 (hi, lo) pairs, two halves per thread (exact
# two-sum of p, plus the FMA residual), then sum the block's pairs as fp32 pairs in a fixed order:
# the thread's two halves, a butterfly over the warp's 32 lanes, a butterfly over the warps' totals,
# and one promotion to double.  A unit whose total lies outside [2^-56, 2^100) is summed again from
# its stored values in double.  The emulation below follows that arithmetic in numpy fp32 (every
# operation correctly rounded, the FMA residual from exact double arithmetic) and checks the claim
# the threshold rests on: inside the range the fast total is within 2^-30 of the exact sum (squares
# that lost bits below 2^-102 cannot move it more), and a unit of only tiny values, or of values
# whose squares overflow fp32, lands outside it.

LO, HI = 2.0 ** -56, 2.0 ** 100
F = np.float32


def _two_sum(a, b):
    s = (a + b).astype(F)
    bb = (s - a).astype(F)
    err = ((a - (s - bb).astype(F)).astype(F) + (b - bb).astype(F)).astype(F)
    return s, err


def _sq_add(a, b):
    """The kernels' pair addition: (s, e) + (s', e') = (fl(s + s'), fl(fl(e + e') + exact error))."""
    s, err = _two_sum(a[0], b[0])
    return s, ((a[1] + b[1]).astype(F) + err).astype(F)


def _butterfly(p, width):
    """xor butterfly over groups of `width` consecutive lanes; every lane ends with its group's total."""
    idx = np.arange(p[0].size)
    o = width // 2
    while o:
        p = _sq_add(p, (p[0][idx ^ o], p[1][idx ^ o]))
        o //= 2
    return p


def _fast_unit_total(values, threads=256):
    """The kernels' fast sum of squares of one unit: half h of thread t takes values 2t + h,
    2t + h + 2*threads, ... (two halves of one f32x2 accumulator per thread)."""
    halves = 2 * threads
    v = np.asarray(values, F)
    per = -(-v.size // halves)
    v = np.concatenate([v, np.zeros(per * halves - v.size, F)]).reshape(per, halves)
    hi = np.zeros(halves, F)
    lo = np.zeros(halves, F)
    with np.errstate(over="ignore", invalid="ignore"):
        for c in v:
            p, pe = _pair(c)
            s, e = _two_sum(hi, p)
            lo = (lo + (e + pe).astype(F)).astype(F)
            hi = s
        t = _sq_add((hi[0::2], lo[0::2]), (hi[1::2], lo[1::2]))  # each thread's two halves
        t = _butterfly(t, 32)                                    # the warp's lanes
        w = (t[0][::32].copy(), t[1][::32].copy())               # lane 0 of each warp
        w = _butterfly(w, w[0].size)                             # the warps' totals
        return float(np.float64(w[0][0]) + np.float64(w[1][0]))


def _exact_sum(values):
    import math

    return math.fsum(float(x) * float(x) for x in np.asarray(values, np.float64))


def test_fast_total_is_close_inside_the_range():
    rng = np.random.default_rng(2)
    inside = 0
    for trial in range(40):
        n = 65536 if trial % 4 == 0 else 4096
        scale = 2.0 ** rng.uniform(-50, 45)
        v = (rng.standard_normal(n) * scale).astype(np.float32)
        k = rng.integers(0, n // 2)  # a share of values below 2^-51, whose squares lose bits
        v[:k] = (rng.standard_normal(k) * 2.0 ** rng.uniform(-80, -52)).astype(np.float32)
        fast, exact = _fast_unit_total(v), _exact_sum(v)
        if LO <= fast < HI:
            inside += 1
            assert abs(fast - exact) <= 2.0 ** -30 * exact, (trial, fast, exact)
    assert inside >= 30  # the draws exercise the range, not only the fallback


def test_tiny_and_huge_units_leave_the_range():
    rng = np.random.default_rng(3)
    for e in (-52, -60, -75, -100, -126):
        v = (rng.standard_normal(4096) * 2.0 ** e).astype(np.float32)
        assert not (LO <= _fast_unit_total(v) < HI), e  # summed again in double
    for e in (50, 60, 64, 100):
        v = (rng.standard_normal(4096) * 2.0 ** e).astype(np.float32)
        t = _fast_unit_total(v)
        assert not (LO <= t < HI), (e, t)  # too large, infinite or NaN: summed again in double


def test_reduction_error_is_far_below_fp32_resolution():
    """With every square exact (all |c| >= 2^-51), only the block's pair reduction rounds: the fast
    total stays within 2^-40 of the exact sum -- for Gaussian units, magnitudes spread over 2^+-20,
    a 1% heavy tail, and strictly positive sums, all inside the exact range -- so a scale rounded to
    fp32 from it almost never differs from the one rounded from the exact sum."""
    rng = np.random.default_rng(11)
    for trial in range(36):
        n = (4096, 65536, 8 * 65536 + 5)[trial % 3]
        kind = trial % 4
        if kind == 0:
            v = rng.standard_normal(n)
        elif kind == 1:
            v = rng.standard_normal(n) * 2.0 ** rng.integers(-20, 20, size=n)
        elif kind == 2:
            v = np.where(rng.random(n) < 0.01, 1e6, 1e-3) * rng.standard_normal(n)
        else:
            v = np.abs(rng.standard_normal(n)) + 1.0
        v = (v * 2.0 ** rng.uniform(-10, 10)).astype(np.float32)
        assert np.all(np.abs(v) >= 2.0 ** -51)  # every square exact
        fast, exact = _fast_unit_total(v), _exact_sum(v)
        assert LO <= fast < HI, trial
        assert abs(fast - exact) <= 2.0 ** -40 * exact, (trial, fast, exact)
