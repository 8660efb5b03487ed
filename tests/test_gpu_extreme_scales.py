"""GPU parity with scales whose product leaves the FP32 range.

scale = amax / 448, so operands whose values all lie near 1e-20 get scales
near 1e-23 and operands near 1e22 scales near 1e20.  The product of two such
scales (1e-46, or 1e40) is not an FP32 number although the outputs
scale_a * scale_b * (A B) can be: the kernels apply the scales one after the
other, (acc * scale_a) * scale_b, and must match the oracle (which forms the
product in fp64) within the bound.

* tiny scales: the codes are large and positive (256 .. 448), so every
  accumulator lies in [K 256^2, K 448^2] and every output in BF16's normal
  range; an FP32 scale product would flush to zero or keep a few bits.
* huge scales: the codes are E4M3 subnormals of both signs (|v| <= 7 2^-9),
  so the outputs stay below the BF16 maximum; an FP32 scale product would
  be infinite.  Rows and columns of zero codes must give exact zeros
  (infinity times zero would give NaN).
"""

import numpy as np
import pytest

import oracle
from _helpers import assert_within_bound, bf16_to_f64, lib, random_codes, to_dev

pytestmark = pytest.mark.gpu

LARGE_CODES = np.arange(0x78, 0x7F, dtype=np.uint8)           # 256 .. 448
SUBNORMAL_CODES = np.concatenate([np.arange(0x01, 0x08), np.arange(0x81, 0x88)]
                                 ).astype(np.uint8)            # +-(1 .. 7) 2^-9

TINY = [(1e-23, 1e-23), (3e-22, 4e-23), (2e-30, 1e-15)]
HUGE = [(1e20, 1e20), (3e25, 2e14)]


def _operands(rng, M, N, K, regime):
    if regime == "tiny":
        return rng.choice(LARGE_CODES, (M, K)), rng.choice(LARGE_CODES, (N, K))
    A = rng.choice(SUBNORMAL_CODES, (M, K))
    B = rng.choice(SUBNORMAL_CODES, (N, K))
    A[3] = 0
    A[M - 2] = 0x80                                            # -0
    B[5] = 0
    return A, B


def _cases():
    for sa, sb in TINY:
        yield "tiny", sa, sb
    for sa, sb in HUGE:
        yield "huge", sa, sb


def _in_range(r):
    """Outputs of the case lie in BF16's normal range (or are exact zeros)."""
    a = np.abs(r)
    return np.all((a == 0) | ((a >= 2.0 ** -126) & (a < 3.3e38)))


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("regime,sa,sb", list(_cases()))
def test_pertensor_gemm_extreme_scales(regime, sa, sb, variant):
    import torch
    fl = lib()
    rng = np.random.default_rng(60 + variant)
    M, N, K = 256, 272, (4096 if regime == "tiny" else 96)
    A, B = _operands(rng, M, N, K, regime)
    sa, sb = np.float32(sa), np.float32(sb)
    fl.fp8la_set_gemm_variant(variant)
    try:
        C = fl.gemm(to_dev(A), to_dev(B), torch.tensor([sa], device="cuda"),
                    torch.tensor([sb], device="cuda"))
        torch.cuda.synchronize()
    finally:
        fl.fp8la_set_gemm_variant(0)
    assert fl.device_status() == 0
    r, _ = oracle.gemm_pertensor(A, B, sa, sb)
    assert _in_range(r), "the case itself leaves the BF16 range"
    got = bf16_to_f64(C)
    what = "%s sa %g sb %g variant %d" % (regime, sa, sb, variant)
    assert_within_bound(got, r, oracle.tolerance_pertensor(A, B, sa, sb, r), what)
    if regime == "huge":
        assert np.all(got[3] == 0) and np.all(got[M - 2] == 0) and np.all(got[:, 5] == 0)


@pytest.mark.parametrize("variant", [1, 2])
def test_grouped_gemm_extreme_scales(variant):
    """Four experts: tiny scales, huge scales, no rows, ordinary scales."""
    import torch
    fl = lib()
    rng = np.random.default_rng(70 + variant)
    E, N, K = 4, 272, 4096
    offs = np.array([0, 130, 300, 300, 400], np.int32)
    sa = np.array([1e-23, 3e25, 1.0, 0.02], np.float32)
    sb = np.array([1e-23, 2e13, 1.0, 1.5], np.float32)
    A = np.zeros((400, K), np.uint8)
    B = np.zeros((E, N, K), np.uint8)
    A[0:130], B[0] = _operands(rng, 130, N, K, "tiny")
    A[130:300], B[1] = _operands(rng, 170, N, K, "huge")
    A[300:400], B[3] = random_codes(rng, (100, K)), random_codes(rng, (N, K))
    d_off, d_sa, d_sb = to_dev(offs), to_dev(sa), to_dev(sb)
    fl.fp8la_set_gemm_variant(variant)
    try:
        C = fl.grouped_gemm(d_off, to_dev(A), to_dev(B), d_sa, d_sb)
        torch.cuda.synchronize()
    finally:
        fl.fp8la_set_gemm_variant(0)
    assert fl.device_status() == 0
    got = bf16_to_f64(C)
    r, _ = oracle.gemm_grouped(A, offs, B, sa, sb)
    for e in (0, 1, 3):
        lo, hi = offs[e], offs[e + 1]
        assert _in_range(r[lo:hi]), "group %d leaves the BF16 range" % e
        assert_within_bound(got[lo:hi], r[lo:hi],
                            oracle.tolerance_pertensor(A[lo:hi], B[e], sa[e], sb[e],
                                                       r[lo:hi]),
                            "variant %d group %d" % (variant, e))
    assert np.all(got[130 + 3] == 0) and np.all(got[130:300, 5] == 0)


def test_blockscaled_gemm_small_normal_scale_products():
    """The block-scaled promotion multiplies each partial sum by the FP32
    product of its two tile scales; with tile scales in [2^-61, 2^-59] those
    products lie in [2^-122, 2^-118], normal FP32 numbers near the bottom of
    the range, and the outputs must still meet the bound."""
    import torch
    fl = lib()
    rng = np.random.default_rng(80)
    M, N, K = 200, 160, 320
    A, B = rng.choice(LARGE_CODES, (M, K)), rng.choice(LARGE_CODES, (N, K))
    A[7, :] = 0
    sa = (2.0 ** rng.uniform(-61, -59, (-(-M // 32), K // 32))).astype(np.float32)
    sb = (2.0 ** rng.uniform(-61, -59, (-(-N // 32), K // 32))).astype(np.float32)
    prod = sa[:, None, :].astype(np.float64) * sb[None, :, :]
    assert prod.min() >= 2.0 ** -126

    def dev_scales(s):
        d = torch.zeros((s.shape[0], (s.shape[1] + 3) // 4 * 4), dtype=torch.float32,
                        device="cuda")
        d[:, :s.shape[1]] = to_dev(s)
        return d[:, :s.shape[1]]

    C = fl.gemm_blockscaled_32x32(to_dev(A), to_dev(B), dev_scales(sa), dev_scales(sb))
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    r, _ = oracle.gemm_blockscaled_32x32(A, B, sa, sb)
    assert _in_range(r)
    got = bf16_to_f64(C)
    assert_within_bound(got, r, oracle.tolerance_blockscaled_32x32(A, B, sa, sb, r),
                        "block-scaled, small tile-scale products")
    assert np.all(got[7] == 0)


@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("sa,sb", [(np.inf, 0.5), (1.0, -np.inf), (np.nan, 1.0), (0.0, 3.0),
                                   (np.inf, 0.0)])
def test_pertensor_gemm_nonfinite_and_zero_scales(sa, sb, variant):
    """A tensor holding +-Inf gets scale Inf from the quantiser.  With a
    non-finite or zero scale every output follows IEEE arithmetic on the
    exact product: +-Inf where the sum is nonzero, NaN where an infinite scale
    meets a zero sum (or a NaN scale), zero for a zero scale.  The GPU must
    give the oracle's value class and sign at every output."""
    import torch
    fl = lib()
    rng = np.random.default_rng(90 + variant)
    M, N, K = 200, 144, 64
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    A[9] = 0                      # zero sums in row 9
    sa, sb = np.float32(sa), np.float32(sb)
    fl.fp8la_set_gemm_variant(variant)
    try:
        C = fl.gemm(to_dev(A), to_dev(B), torch.tensor([sa], device="cuda"),
                    torch.tensor([sb], device="cuda"))
        torch.cuda.synchronize()
    finally:
        fl.fp8la_set_gemm_variant(0)
    assert fl.device_status() == 0
    with np.errstate(invalid="ignore"):
        r, _ = oracle.gemm_pertensor(A, B, sa, sb)
    got = bf16_to_f64(C)
    assert np.array_equal(np.isnan(got), np.isnan(r))
    fin = ~np.isnan(r)
    assert np.all(np.isinf(r[fin]) | (r[fin] == 0)), "the case has other outputs"
    assert np.array_equal(got[fin], r[fin])      # +-Inf with the oracle's sign, or 0
