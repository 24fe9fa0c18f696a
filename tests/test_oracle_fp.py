"""Pins for the oracle's exact fp32/fp16 helpers (CPU only).

The fused multiply-add emulation is checked against exact rational
arithmetic with correct rounding to fp32, not against a re-typed formula.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import fp


def _round_f32_exact(x: Fraction) -> np.float32:
    """Correctly rounded fp32 of an exact rational (ties to even)."""
    r0 = np.float32(float(x))
    cands = [r0, np.nextafter(r0, np.float32(np.inf)), np.nextafter(r0, np.float32(-np.inf))]
    best = None
    for c in cands:
        if not np.isfinite(c):
            continue
        dist = abs(Fraction(float(c)) - x)
        key = (dist, int(np.frombuffer(np.float32(c).tobytes(), np.uint32)[0]) & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return np.float32(best[1])


def _exact_fma(a, b, c):
    return _round_f32_exact(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


def test_fma_random_matches_exact_rounding():
    rng = np.random.default_rng(1)
    a = rng.standard_normal(3000).astype(np.float32)
    b = rng.standard_normal(3000).astype(np.float32)
    c = (rng.standard_normal(3000) * 10.0 ** rng.integers(-6, 6, 3000)).astype(np.float32)
    got = fp.fma_f32(a, b, c)
    for i in range(3000):
        assert got[i] == _exact_fma(a[i], b[i], c[i]), i


def test_fma_adversarial_midpoints():
    # a*b lands half an ulp off an fp32 value plus a tiny c: plain fp64
    # evaluation followed by rounding to fp32 would break the tie wrongly.
    cases = []
    one = np.float32(1.0)
    half_ulp = 2.0 ** -24
    a = np.float32(1.0 + 2.0 ** -12)
    b = np.float32(1.0 + 2.0 ** -12)      # a*b = 1 + 2^-11 + 2^-24 exactly
    cases.append((a, b, np.float32(0.0)))
    cases.append((a, b, np.float32(2.0 ** -60)))
    cases.append((a, b, np.float32(-2.0 ** -60)))
    cases.append((one, np.float32(1.0 + 2.0 ** -23), np.float32(half_ulp)))
    cases.append((one, np.float32(1.0), np.float32(half_ulp)))
    cases.append((np.float32(3.0), np.float32(1.0 / 3.0), np.float32(-1.0)))
    rng = np.random.default_rng(7)
    for _ in range(400):
        x = np.float32(rng.standard_normal())
        y = np.float32(rng.standard_normal())
        p = Fraction(float(x)) * Fraction(float(y))
        # c = -(nearest fp32 to p): heavy cancellation
        cases.append((x, y, np.float32(-float(p))))
    for a, b, c in cases:
        assert fp.fma_f32(a, b, c) == _exact_fma(a, b, c), (a, b, c)


def test_chain_matvec_exact_on_integers_and_bounded_otherwise():
    rng = np.random.default_rng(3)
    x = rng.integers(-50, 50, size=(5, 16)).astype(np.float32)
    m = rng.integers(-50, 50, size=(16, 7)).astype(np.float32)
    assert np.array_equal(fp.chain_matvec_f32(x, m), (x.astype(np.int64) @ m.astype(np.int64)).astype(np.float32))
    x = rng.standard_normal((4, 128)).astype(np.float32)
    m = rng.standard_normal((128, 128)).astype(np.float32)
    got = fp.chain_matvec_f32(x, m).astype(np.float64)
    exact = x.astype(np.float64) @ m.astype(np.float64)
    bound = 128 * 2.0 ** -24 * (np.abs(x).astype(np.float64) @ np.abs(m).astype(np.float64))
    assert np.all(np.abs(got - exact) <= bound)


def test_chain_sumsq():
    x = np.arange(1, 11, dtype=np.float32)[None, :]
    assert fp.chain_sumsq_f32(x)[0] == np.float32(385.0)


@pytest.mark.parametrize("x,expect", [
    (1.0 + 2.0 ** -11, 1.0),                     # tie -> even
    (1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -9),     # tie -> even (up)
    (1.0 + 2.0 ** -11 + 2.0 ** -20, 1.0 + 2.0 ** -10),
    (65504.0, 65504.0),
    (65519.0, 65504.0),                          # rounds down to max
    (65520.0, 65504.0),                          # would overflow: saturates
    (-1e9, -65504.0),
    (2.0 ** -24, 2.0 ** -24),                    # smallest subnormal
    (2.0 ** -26, 0.0),
])
def test_f16_rounding_and_saturation(x, expect):
    assert float(fp.f16_rn_sat(np.float32(x))) == expect
