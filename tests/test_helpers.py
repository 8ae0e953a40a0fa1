"""Pins of the test helpers that stand for a rounding of the kernels."""
import numpy as np

from _helpers import rna_tf32


def test_rna_tf32_nearest_ties_away():
    """10 stored mantissa bits: 1 + 2^-11 lies halfway between 1 and
    1 + 2^-10 and rounds away from zero, on both signs; just below the
    midpoint rounds down; the result is the nearest value with the 13 low
    bits clear, which a direct search over the two neighbours confirms."""
    one = np.float32(1.0)
    assert rna_tf32(np.float32(1 + 2.0 ** -11)) == 1 + 2.0 ** -10
    assert rna_tf32(np.float32(-(1 + 2.0 ** -11))) == -(1 + 2.0 ** -10)
    assert rna_tf32(np.nextafter(np.float32(1 + 2.0 ** -11), one)) == 1.0
    assert rna_tf32(np.float32(3 * 2.0 ** -11 + 1)) == 1 + 2.0 ** -9  # tie between odd and even: away
    x = np.random.default_rng(0).standard_normal(20000).astype(np.float32) * 10.0 ** np.random.default_rng(1).integers(-20, 20, 20000)
    r = rna_tf32(x)
    assert np.all(r.astype(np.float32).view(np.uint32) & 0x1FFF == 0)
    m, e = np.frexp(x.astype(np.float64))
    lo = np.ldexp(np.floor(np.abs(m) * 2048.0), e - 11) * np.sign(m)
    hi = lo + np.ldexp(1.0, e - 11) * np.sign(m)
    near = np.where(np.abs(x - lo) < np.abs(hi - x), lo, hi)  # ties (equal distance) go to hi, away from zero
    assert np.array_equal(r, near)
    assert np.all(np.abs(r - x) <= 2.0 ** -11 * np.abs(x))
