"""Pins for the oracle's E4M3 decode and encode (CPU only).

What pins them, none of it the oracle's own code: hand-worked values of the
published format (tests/golden/e4m3_values.json), the format's fixed
invariants, PyTorch's float8_e4m3fn CPU conversion (a library routine), and
exact rational arithmetic for rounding decisions.
"""

import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    with open(os.path.join(GOLDEN, "e4m3_values.json")) as f:
        return json.load(f)


def test_decode_hand_values():
    g = _golden()
    for code, val in g["values"].items():
        got = oracle.decode_code(int(code, 16))
        assert got == val, code
        assert np.signbit(got) == np.signbit(val), code
    for code in g["nan_codes"]:
        assert np.isnan(oracle.decode_code(int(code, 16)))


def test_decode_invariants():
    vals = oracle.decode(np.arange(256, dtype=np.uint8))
    pos = vals[:0x7F]
    # strictly increasing magnitudes over 0x00..0x7E
    assert np.all(np.diff(pos) > 0)
    assert pos.max() == 448.0 == oracle.E4M3_MAX
    assert np.count_nonzero(pos > 0) == _golden()["count_finite_positive_nonzero"]
    # sign symmetry: code | 0x80 is the negation
    assert np.array_equal(vals[0x80:0xFF], -vals[:0x7F])
    # exactly two NaN codes, no infinities
    assert np.flatnonzero(np.isnan(vals)).tolist() == [0x7F, 0xFF]
    assert not np.any(np.isinf(vals))
    # subnormal spacing 2^-9, normal binade [2^-6, 2^-5) spacing 2^-9 too
    assert np.all(np.diff(pos[:16]) == 2.0 ** -9)


def test_decode_matches_torch_float8_e4m3fn():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def _dec_frac(c):
    """Exact rational value of a finite code, from its bit fields."""
    s, e, m = (c >> 7) & 1, (c >> 3) & 15, c & 7
    v = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -v if s else v


def test_encode_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.decode(codes).astype(np.float32)
    assert np.array_equal(oracle.encode(vals), codes)


def test_encode_midpoints_go_to_even():
    for c in range(0x7E):
        lo, hi = _dec_frac(c), _dec_frac(c + 1)
        mid = (lo + hi) / 2
        x = np.float32(float(mid))
        assert Fraction(float(x)) == mid          # every midpoint fits in fp32
        even = c if c % 2 == 0 else c + 1
        assert oracle.encode(np.array([x]))[0] == even, hex(c)
        assert oracle.encode(np.array([-x]))[0] == even | 0x80, hex(c)
        # one fp32 ulp either side goes to the nearer code
        below = np.nextafter(x, np.float32(0))
        above = np.nextafter(x, np.float32(np.inf))
        assert oracle.encode(np.array([below]))[0] == c
        assert oracle.encode(np.array([above]))[0] == c + 1


def test_encode_saturates_and_specials():
    x = np.array([448.0, 448.0001, 464.0, 500.0, 1e30, np.inf,
                  -448.0001, -np.inf, np.nan, -np.nan, 0.0, -0.0,
                  2.0 ** -10, -(2.0 ** -10), 2.0 ** -11, -1e-30, 1e-45],
                 dtype=np.float32)
    want = [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E,
            0xFE, 0xFE, 0x7F, 0x7F, 0x00, 0x80,
            0x00, 0x80, 0x00, 0x80, 0x00]
    assert oracle.encode(x).tolist() == want


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(1234)
    bits = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) <= 448.0)]
    # add a dense sweep of the normal range too
    x = np.concatenate([x, np.linspace(-448, 448, 200_001, dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.encode(x)
    assert np.array_equal(ref, got)


def test_encode_nearest_by_exact_arithmetic():
    """Brute force: encode(x) is a nearest code by exact rational distance."""
    rng = np.random.default_rng(7)
    xs = (rng.standard_normal(3000) * rng.choice([1e-3, 0.1, 10, 300], 3000)).astype(np.float32)
    finite = [(c, _dec_frac(c)) for c in range(0x7F)]
    for x in xs:
        code = int(oracle.encode(np.array([x]))[0])
        fx = Fraction(float(x))
        if abs(fx) > 448:
            assert code & 0x7F == 0x7E
            continue
        d = abs(abs(fx) - _dec_frac(code & 0x7F))
        best = min(abs(abs(fx) - v) for _, v in finite)
        assert d == best
        assert (code >> 7) == (1 if np.signbit(x) else 0)


def _encode_pins_pass(encode):
    """The encoder pins above, as one predicate over an encode function."""
    try:
        codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
        if not np.array_equal(encode(oracle.decode(codes).astype(np.float32)), codes):
            return False
        for c in range(0x7E):
            mid = np.float32(float((_dec_frac(c) + _dec_frac(c + 1)) / 2))
            if encode(np.array([mid]))[0] != (c if c % 2 == 0 else c + 1):
                return False
        x = np.array([500.0, -np.inf, -0.0, np.nan], dtype=np.float32)
        return encode(x).tolist() == [0x7E, 0xFE, 0x80, 0x7F]
    except Exception:
        return False


def _mutant(kind):
    def enc(x):
        x = np.asarray(x, dtype=np.float32)
        if kind == "ties_away":
            # nudge exact midpoints upward: ties round away from zero
            up = np.nextafter(np.abs(x), np.float32(np.inf)) * np.sign(x)
            mids = set(float((_dec_frac(c) + _dec_frac(c + 1)) / 2) for c in range(0x7E))
            x = np.array([u if abs(float(v)) in mids else v for v, u in zip(x.ravel(), up.ravel())],
                         dtype=np.float32).reshape(x.shape)
            return oracle.encode(x)
        if kind == "no_saturation":
            out = oracle.encode(x)
            return np.where(np.abs(x) > 464, np.uint8(0x7F), out).astype(np.uint8)
        if kind == "sign_of_zero_dropped":
            out = oracle.encode(x)
            return np.where(out == 0x80, np.uint8(0), out).astype(np.uint8)
        raise ValueError(kind)
    return enc


def test_encode_pins_pass_on_oracle():
    assert _encode_pins_pass(oracle.encode)


@pytest.mark.parametrize("kind", ["ties_away", "no_saturation", "sign_of_zero_dropped"])
def test_planted_encoder_mistakes_are_caught(kind):
    assert not _encode_pins_pass(_mutant(kind))


def test_encode_is_monotone_and_odd():
    """Rounding to the nearest code never reverses order, and enc(-x) is
    enc(x) with the sign bit set: checked on sorted random fp32 values that
    span the subnormals, every binade and the saturated range."""
    rng = np.random.default_rng(7)
    mags = np.exp2(rng.uniform(-14.0, 12.0, 200000)).astype(np.float32)
    x = np.sort(mags)
    vals = oracle.decode(oracle.encode(x))
    assert np.all(np.diff(vals) >= 0)
    assert np.array_equal(oracle.encode(-x), oracle.encode(x) | np.uint8(0x80))
