"""Pins for the oracle's GEMM error bound (CPU only).

The bound is |C_gpu - C_ref| <= 2^-8 |C_ref| + 2^-22 K sa sb max|a| max|b|
(FP32 accumulation and one BF16 rounding; page [P1] "通过 CUTLASS 命名约定在
Triton 中实现 FP8 GEMM 内核", optimisation parameter list), and for 32x32
block scales sa max|a| becomes max |sa[m/32][k/32] dec(a)| (page [P3] "JAX 中
使用 Triton 优化 Blackwell GPU 的 FP8 GEMM 内核", implementation paragraph).

Pins: hand-worked values of the formula (tests/golden/bound_cases.json) on
cases built so that each plausible mistake changes the value -- a wrong power
of two, a dropped K, a maximum over raw byte codes instead of decoded values,
max|s| * max|a| in place of max|s*a|, a transposed scale grid, a bound without
the absolute value, a bound taken around the BF16-rounded reference.  Each of
those mistakes is planted below and must fail the pins.  A last test checks
that the GPU tests' comparison rejects an output one BF16 step beyond the
bound and accepts the correctly rounded one.
"""

import json
import os

import numpy as np
import pytest

import oracle
from _helpers import assert_within_bound

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load():
    with open(os.path.join(GOLDEN, "bound_cases.json")) as f:
        return json.load(f)


def _codes(rows):
    return np.array([[int(v, 16) for v in row] for row in rows], dtype=np.uint8)


def _sparse(shape, entries):
    a = np.zeros(shape, dtype=np.uint8)
    for (i, j, v) in entries:
        a[i, j] = int(v, 16)
    return a


def _pins(tol_pt, tol_bs, max_dec=oracle.max_abs_decoded,
          max_ts=oracle.max_abs_tile_scaled_32x32):
    """True when the given bound functions reproduce every hand-worked value."""
    g = _load()
    try:
        for c in g["pertensor"]:
            A, B = _codes(c["A"]), _codes(c["B"])
            sa, sb = np.float32(c["scale_a"]), np.float32(c["scale_b"])
            r, _ = oracle.gemm_pertensor(A, B, sa, sb)
            if not np.array_equal(r, np.array(c["exact"])):
                return False
            if max_dec(A) != c["max_a"] or max_dec(B) != c["max_b"]:
                return False
            if not np.array_equal(tol_pt(A, B, sa, sb, r), np.array(c["bound"])):
                return False
        for c in g["blockscaled"]:
            A = _sparse((c["M"], c["K"]), c["A_nonzero"])
            B = _sparse((c["N"], c["K"]), c["B_nonzero"])
            sa = np.array(c["sa"], dtype=np.float32)
            sb = np.array(c["sb"], dtype=np.float32)
            if max_ts(A, sa) != c["max_sa_a"] or max_ts(B, sb) != c["max_sb_b"]:
                return False
            r, _ = oracle.gemm_blockscaled_32x32(A, B, sa, sb)
            pts = tuple(np.array(c["points"]).T)
            if not np.array_equal(r[pts], np.array(c["exact"])):
                return False
            if not np.array_equal(tol_bs(A, B, sa, sb, r)[pts], np.array(c["bound"])):
                return False
        return True
    except Exception:
        return False


def test_bound_pins_pass():
    assert _pins(oracle.tolerance_pertensor, oracle.tolerance_blockscaled_32x32)


# ------------------------------------------------------------ planted mistakes
def _pt(coef=2.0 ** -22, use_k=True, absval=True, around_bf16=False, maxf=None):
    def f(A, B, sa, sb, r):
        K = A.shape[1] if use_k else 1
        mf = maxf or oracle.max_abs_decoded
        ref = oracle.bf16_bits_to_float(oracle.bf16_rne(r)) if around_bf16 else r
        first = (2.0 ** -8) * (np.abs(ref) if absval else ref)
        return first + coef * K * float(np.float32(sa)) * float(np.float32(sb)) * mf(A) * mf(B)
    return f


def _bs(coef=2.0 ** -22, use_k=True, maxf=None):
    def f(A, B, sa, sb, r):
        K = A.shape[1] if use_k else 1
        mf = maxf or oracle.max_abs_tile_scaled_32x32
        return (2.0 ** -8) * np.abs(r) + coef * K * mf(A, sa) * mf(B, sb)
    return f


def _raw_max(codes):
    return float(np.asarray(codes, dtype=np.float64).max())


def _raw_tile_max(codes, s):
    M, K = codes.shape
    s = np.asarray(s, dtype=np.float64)
    return float((np.abs(s[np.arange(M) // 32][:, np.arange(K) // 32])
                  * codes.astype(np.float64)).max())


def _separate_maxima(codes, s):
    return float(np.abs(np.asarray(s, dtype=np.float64)).max()
                 * oracle.max_abs_decoded(codes))


def _transposed_grid(codes, s):
    M, K = codes.shape
    s = np.asarray(s, dtype=np.float64)
    tiles = max(M, K) // 32 + 1
    g = np.zeros((tiles, tiles))
    g[:s.shape[1], :s.shape[0]] = np.abs(s).T         # s read as s[k/32][m/32]
    w = g[np.arange(M) // 32][:, np.arange(K) // 32] * np.abs(oracle.decode(codes))
    return float(w.max())


MUTANTS = {
    "coefficient 2^-20": (_pt(coef=2.0 ** -20), _bs(coef=2.0 ** -20)),
    "K dropped (per tensor)": (_pt(use_k=False), oracle.tolerance_blockscaled_32x32),
    "K dropped (block)": (oracle.tolerance_pertensor, _bs(use_k=False)),
    "no absolute value of C_ref": (_pt(absval=False), oracle.tolerance_blockscaled_32x32),
    "bound around bf16(r)": (_pt(around_bf16=True), oracle.tolerance_blockscaled_32x32),
    "max over raw codes (per tensor)": (_pt(maxf=_raw_max), oracle.tolerance_blockscaled_32x32),
    "max over raw codes (block)": (oracle.tolerance_pertensor, _bs(maxf=_raw_tile_max)),
    "max|s| * max|a| (block)": (oracle.tolerance_pertensor, _bs(maxf=_separate_maxima)),
    "transposed scale grid (block)": (oracle.tolerance_pertensor, _bs(maxf=_transposed_grid)),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_bound_mistakes_are_caught(name):
    tol_pt, tol_bs = MUTANTS[name]
    assert not _pins(tol_pt, tol_bs)


def test_planted_max_mistakes_are_caught():
    assert not _pins(oracle.tolerance_pertensor, oracle.tolerance_blockscaled_32x32,
                     max_dec=_raw_max)
    assert not _pins(oracle.tolerance_pertensor, oracle.tolerance_blockscaled_32x32,
                     max_ts=_separate_maxima)


# --------------------------------------------- the comparison the GPU tests use
def _bf16_neighbour(x, steps):
    """The BF16 value `steps` representable steps away from BF16 value x."""
    bits = np.float32(x).view(np.uint32) >> 16
    sign = bits & 0x8000
    mag = (bits & 0x7FFF).astype(np.int64)
    # walk along the real line: for negative x a step up lowers the magnitude
    mag = mag + (steps if sign == 0 else -steps)
    if mag < 0:
        sign, mag = sign ^ 0x8000, -mag
    out = np.uint32((sign | mag) << 16).view(np.float32)
    return float(out)


def _first_beyond(r, bound, direction):
    """First BF16 value on the given side of r that lies outside the bound."""
    c = float(oracle.bf16_bits_to_float(oracle.bf16_rne(np.array([r])))[0])
    while abs(c - r) <= bound:
        c = _bf16_neighbour(c, direction)
    return c


@pytest.mark.parametrize("kind", ["pertensor", "blockscaled"])
def test_comparison_rejects_one_bf16_step_beyond_the_bound(kind):
    rng = np.random.default_rng(61)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    if kind == "pertensor":
        A, B = rng.choice(finite, (24, 96)), rng.choice(finite, (20, 96))
        sa, sb = np.float32(0.013), np.float32(2.5)
        r, C = oracle.gemm_pertensor(A, B, sa, sb)
        bound = oracle.tolerance_pertensor(A, B, sa, sb, r)
    else:
        A, B = rng.choice(finite, (70, 100)), rng.choice(finite, (45, 100))
        sa = rng.uniform(0.01, 3, (3, 4)).astype(np.float32)
        sb = rng.uniform(0.01, 3, (2, 4)).astype(np.float32)
        r, C = oracle.gemm_blockscaled_32x32(A, B, sa, sb)
        bound = oracle.tolerance_blockscaled_32x32(A, B, sa, sb, r)
    good = oracle.bf16_bits_to_float(C)
    assert_within_bound(good, r, bound, kind)          # the rounded reference passes
    for idx in [(0, 0), (5, 7), (r.shape[0] - 1, r.shape[1] - 1)]:
        for direction in (+1, -1):
            bad = good.copy()
            bad[idx] = _first_beyond(r[idx], bound[idx], direction)
            # the replaced value is at most one BF16 step past the bound's edge
            inner = _bf16_neighbour(bad[idx], -direction)
            assert abs(inner - r[idx]) <= bound[idx]
            with pytest.raises(AssertionError):
                assert_within_bound(bad, r, bound, kind)
    nan = good.copy()
    nan[1, 1] = np.nan
    with pytest.raises(AssertionError):
        assert_within_bound(nan, r, bound, kind)
