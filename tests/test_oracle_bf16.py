"""Pins for the oracle's fp64 -> bf16 round-to-nearest-even (CPU only).

Pins: PyTorch's fp32 -> bfloat16 CPU cast (RNE, a library routine) on values
that are exact in fp32; exact rational rounding (fractions) on fp64 values
that are not, where one direct rounding differs from rounding through fp32;
and the format's fixed values (max, min subnormal, overflow to infinity).
"""

from fractions import Fraction

import numpy as np
import torch

import oracle


def _bits_torch(x32):
    return torch.from_numpy(np.asarray(x32, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_matches_torch_on_fp32_values():
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2 ** 32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    got = oracle.bf16_rne(x.astype(np.float64))
    assert np.array_equal(got, _bits_torch(x))


def _rne_fraction(q):
    """bf16 RNE of an exact rational, independent of the oracle's method."""
    if q == 0:
        return Fraction(0)
    s = -1 if q < 0 else 1
    a = abs(q)
    e = 0
    while a >= Fraction(2) ** (e + 1):
        e += 1
    while a < Fraction(2) ** e:
        e -= 1
    quantum = Fraction(2) ** max(e - 7, -133)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return s * fl * quantum


def test_direct_rounding_not_double_rounding():
    # 1 + 2^-8 + 2^-30: through fp32 it becomes the tie 1 + 2^-8 and then 1.0;
    # rounded once it is just above the midpoint and goes up to 1 + 2^-7.
    r = 1.0 + 2.0 ** -8 + 2.0 ** -30
    got = oracle.bf16_bits_to_float(oracle.bf16_rne(np.array([r])))[0]
    assert got == 1.0 + 2.0 ** -7 == float(_rne_fraction(Fraction(r)))


def test_matches_exact_rationals_on_fp64():
    rng = np.random.default_rng(11)
    r = rng.standard_normal(20000) * np.exp2(rng.integers(-140, 120, 20000))
    got = oracle.bf16_bits_to_float(oracle.bf16_rne(r))
    for x, g in zip(r, got):
        assert g == float(_rne_fraction(Fraction(float(x))))


def test_fixed_values():
    bmax = (2 - 2.0 ** -7) * 2.0 ** 127
    half_ulp = 2.0 ** (127 - 8)
    cases = [
        (0.0, 0x0000), (-0.0, 0x8000), (1.0, 0x3F80), (-2.0, 0xC000),
        (bmax, 0x7F7F), (bmax + half_ulp, 0x7F80),          # tie at max+half ulp overflows
        (np.nextafter(bmax + half_ulp, 0), 0x7F7F),
        (2.0 ** -133, 0x0001), (2.0 ** -134, 0x0000),        # tie to even zero
        (3 * 2.0 ** -135, 0x0001), (-(2.0 ** -200), 0x8000),
        (np.inf, 0x7F80), (-np.inf, 0xFF80),
    ]
    for r, want in cases:
        assert int(oracle.bf16_rne(np.array([r]))[0]) == want, r
    assert int(oracle.bf16_rne(np.array([np.nan]))[0]) == 0x7FC0
