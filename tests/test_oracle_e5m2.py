"""Pins for the oracle's E5M2 decode and encode, and for the E5M2 paths of
the quantiser and the GEMM (CPU only).

Pins: hand-worked values of the format, its invariants, PyTorch's
float8_e5m2 CPU conversion on the range where it cannot overflow (a library
routine), exact rational arithmetic for rounding and for small GEMMs.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import e5m2


def _dec_frac(c):
    s, e, m = (c >> 7) & 1, (c >> 2) & 31, c & 3
    v = Fraction(m, 4) * Fraction(1, 2 ** 14) if e == 0 else (1 + Fraction(m, 4)) * Fraction(2) ** (e - 15)
    return -v if s else v


def test_hand_values():
    # s eeeee mm
    assert e5m2.decode_code(0x3C) == 1.0          # 0 01111 00
    assert e5m2.decode_code(0x3D) == 1.25         # 0 01111 01
    assert e5m2.decode_code(0x40) == 2.0          # 0 10000 00
    assert e5m2.decode_code(0x7B) == 57344.0      # 0 11110 11 = 1.75 * 2^15
    assert e5m2.decode_code(0x04) == 2.0 ** -14   # smallest normal
    assert e5m2.decode_code(0x01) == 2.0 ** -16   # smallest subnormal
    assert e5m2.decode_code(0x7C) == float("inf")
    assert e5m2.decode_code(0xFC) == -float("inf")
    assert all(np.isnan(e5m2.decode_code(c)) for c in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF))
    assert e5m2.decode_code(0xBC) == -1.0
    assert np.signbit(e5m2.decode_code(0x80))


def test_decode_matches_torch_float8_e5m2():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e5m2).to(torch.float64).numpy()
    got = e5m2.decode(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_encode_roundtrip_and_ties():
    finite = np.array([c for c in range(256) if (c & 0x7C) != 0x7C], dtype=np.uint8)
    assert np.array_equal(e5m2.encode(e5m2.decode(finite).astype(np.float32)), finite)
    for c in range(0x7B):
        mid = (_dec_frac(c) + _dec_frac(c + 1)) / 2
        x = np.float32(float(mid))
        assert Fraction(float(x)) == mid
        even = c if c % 2 == 0 else c + 1
        assert e5m2.encode(np.array([x]))[0] == even
        assert e5m2.encode(np.array([np.nextafter(x, np.float32(0))]))[0] == c
        assert e5m2.encode(np.array([np.nextafter(x, np.float32(np.inf))]))[0] == c + 1


def test_encode_saturates_and_specials():
    x = np.array([57344.0, 61439.0, 61440.0, 1e30, np.inf, -np.inf, np.nan, -0.0, 2.0 ** -17],
                 dtype=np.float32)
    assert e5m2.encode(x).tolist() == [0x7B, 0x7B, 0x7B, 0x7B, 0x7B, 0xFB, 0x7F, 0x80, 0x00]


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(77)
    bits = rng.integers(0, 2 ** 32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) <= 57344.0)]
    ref = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(ref, e5m2.encode(x))


def test_quantize_e5m2_amax_lands_on_max_code():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal(1000) * 3).astype(np.float32)
    q, amax, scale = oracle.quantize_pertensor(x, fmt="e5m2")
    assert scale == np.float32(amax) / np.float32(57344.0)
    assert q[int(np.argmax(np.abs(x)))] & 0x7F == 0x7B
    # dequantised error: 2 mantissa bits -> half-step 2^-3 relative (normals)
    y = e5m2.decode(q) * float(scale)
    assert np.all(np.abs(y - x) <= 2.0 ** -3 * np.abs(x) * (1 + 1e-6) + 2.0 ** -17 * float(scale))


@pytest.mark.parametrize("fa,fb", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
def test_gemm_formats_exact_rational(fa, fb):
    rng = np.random.default_rng(5)
    finite5 = np.array([c for c in range(256) if (c & 0x7C) != 0x7C], dtype=np.uint8)
    finite4 = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    pick = {"e5m2": finite5, "e4m3": finite4}
    dec = {"e5m2": _dec_frac,
           "e4m3": lambda c: (lambda s, e, m: (-1 if s else 1) * (Fraction(m, 8) / 64 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)))((c >> 7) & 1, (c >> 3) & 15, c & 7)}
    M, N, K = 3, 2, 5
    A = rng.choice(pick[fa], size=(M, K)).astype(np.uint8)
    B = rng.choice(pick[fb], size=(N, K)).astype(np.uint8)
    r, C = oracle.gemm_pertensor(A, B, 0.5, 0.25, a_fmt=fa, b_fmt=fb)
    for m in range(M):
        for n in range(N):
            q = Fraction(1, 8) * sum(dec[fa](int(A[m, k])) * dec[fb](int(B[n, k])) for k in range(K))
            # E5M2 sums may round in fp64 at 2^-53 relative
            assert abs(Fraction(float(r[m, n])) - q) <= abs(q) * Fraction(1, 2 ** 50)


def test_encode_is_monotone_and_odd():
    """As for E4M3: order-preserving and sign-symmetric rounding, over the
    subnormals, every binade and the saturated range of E5M2."""
    rng = np.random.default_rng(8)
    x = np.sort(np.exp2(rng.uniform(-20.0, 18.0, 200000)).astype(np.float32))
    vals = e5m2.decode(e5m2.encode(x))
    assert np.all(np.diff(vals) >= 0)
    assert np.array_equal(e5m2.encode(-x), e5m2.encode(x) | np.uint8(0x80))
