"""The kernels take the reciprocal of each softmax denominator d (at most 256
terms, the largest 1 or within a few ulp of it: d in [2^-8, 2^8]) by one Newton-Raphson
correction, in Markstein's fused form, of a hardware seed y within one ulp of 1/d:
r = fma(-d, y, 1); y1 = fma(y, r, y); and when the significand of d is all ones the
lowest bit of y1 is set.  The claim is that this equals the IEEE round-to-nearest
1/d for EVERY seed within one ulp.  Here it is checked exhaustively over the binade
[1, 2) with exact emulation of the two fused operations, and on samples of every
other binade from 2^-8 to 2^8 (the step commutes with scaling by 2^k there).

The fused operations are emulated exactly: d*y has 48 significant bits and is
exact in float64, so 1 - d*y (|r| < 2^-22) is exact too and rounding it to
float32 is the FMA's single rounding; y*r is exact in float64, and y + y*r is
carried as an exact (hi, lo) pair (TwoSum) before the one rounding to float32.
"""
import numpy as np


def _two_sum(a, b):
    s = a + b
    bb = s - a
    return s, (a - (s - bb)) + (b - bb)


def _round32(hi, lo):
    """float32 round-to-nearest-even of the exact value hi + lo, hi = fl64(hi + lo).
    float32 midpoints are float64 numbers, so fl32(hi) is right unless hi sits
    exactly on a midpoint, where the sign of lo decides."""
    c = hi.astype(np.float32)
    c64 = c.astype(np.float64)
    up = np.nextafter(c, np.float32(np.inf))
    dn = np.nextafter(c, np.float32(-np.inf))
    on_up = hi == (c64 + up.astype(np.float64)) / 2
    on_dn = hi == (c64 + dn.astype(np.float64)) / 2
    c = np.where(on_up & (lo > 0), up, c)
    return np.where(on_dn & (lo < 0), dn, c)


def _step(d, y):
    d64, y64 = d.astype(np.float64), y.astype(np.float64)
    r = (1.0 - d64 * y64).astype(np.float32)
    hi, lo = _two_sum(y64, y64 * r.astype(np.float64))
    y1 = _round32(hi, lo)
    tie = (~d.view(np.uint32) & np.uint32(0x7FFFFF)) == 0
    return np.where(tie, (y1.view(np.uint32) | np.uint32(1)).view(np.float32), y1)


def _check(d):
    want = np.float32(1) / d                       # IEEE round to nearest
    q = 1.0 / d.astype(np.float64)
    ulp = np.spacing(want).astype(np.float64)
    a = q.astype(np.float32)
    n_seeds = 0
    for y in (np.nextafter(a, np.float32(0)), a, np.nextafter(a, np.float32(4))):
        ok = np.abs(y.astype(np.float64) - q) < ulp  # the seeds the hardware may return
        got = _step(d, y)
        bad = ok & (got != want)
        assert not bad.any(), (d[bad][:4], y[bad][:4], got[bad][:4], want[bad][:4])
        n_seeds += int(ok.sum())
    return n_seeds


def test_reciprocal_step_exhaustive_over_one_binade():
    total = 0
    for lo in range(0, 1 << 23, 1 << 21):
        bits = np.arange(lo, lo + (1 << 21), dtype=np.uint32) + np.uint32(0x3F800000)
        total += _check(bits.view(np.float32))
    assert total >= 2 * (1 << 23) - 16  # two seeds per d (almost everywhere)


def test_reciprocal_step_other_binades_sampled():
    rng = np.random.default_rng(7)
    for k in list(range(-8, 0)) + list(range(1, 8)):  # [2^-8, 2^-7) ... [128, 256)
        m = rng.integers(0, 1 << 23, 200000, dtype=np.uint32)
        m[:3] = (0, 1, (1 << 23) - 1)
        d = (m | np.uint32((127 + k) << 23)).view(np.float32)
        _check(d)
    _check(np.array([256.0], dtype=np.float32))


def test_reciprocal_step_without_the_tie_fix_fails_once_per_binade():
    """The all-ones significand is the one place the bare step goes wrong: the
    seed 2^-(k+1) lands on a rounding tie that ties-to-even resolves downwards."""
    d = np.array([np.nextafter(np.float32(2), np.float32(0))], dtype=np.float32)
    y = np.array([0.5], dtype=np.float32)
    d64, y64 = d.astype(np.float64), y.astype(np.float64)
    r = (1.0 - d64 * y64).astype(np.float32)
    hi, lo = _two_sum(y64, y64 * r.astype(np.float64))
    assert _round32(hi, lo)[0] == np.float32(0.5) != np.float32(1) / d[0]
    assert _step(d, y)[0] == np.float32(1) / d[0]
