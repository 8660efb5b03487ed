"""GPU parity with NaN operand codes.

E4M3 has one NaN pattern per sign, S.1111.111 (0x7F, 0xFF); its decoded
value is NaN, and a NaN product makes every sum it enters NaN (NaN x 0 is
NaN).  So a NaN code in row m of A makes output row m NaN, and a NaN code in
row n of B (output column n) makes that column NaN.  The oracle computes
exactly that; the GPU outputs must be NaN at the same places and within the
bound everywhere else (the bound's maxima leave NaN codes out).
"""

import numpy as np
import pytest

import oracle
from _helpers import assert_within_bound, bf16_to_f64, lib, random_codes, to_dev

pytestmark = pytest.mark.gpu


def _check(got, r, bound, what):
    nan_ref = np.isnan(r)
    assert nan_ref.any(), what + ": the case has no NaN outputs"
    assert np.array_equal(np.isnan(got), nan_ref), what + ": NaN outputs differ"
    keep = ~nan_ref.any(axis=1)
    assert_within_bound(got[keep][:, ~nan_ref.any(axis=0)],
                        r[keep][:, ~nan_ref.any(axis=0)],
                        bound[keep][:, ~nan_ref.any(axis=0)], what)


def _codes_with_nans(rng, M, N, K):
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    A[5, 10] = 0x7F
    A[M - 1, K - 1] = 0xFF
    B[7, 3] = 0x7F
    return A, B


@pytest.mark.parametrize("variant", [0, 1, 2, 3])
def test_pertensor_gemm_nan_codes(variant):
    import torch
    fl = lib()
    rng = np.random.default_rng(40 + variant)
    M, N, K = 300, 260, 96
    A, B = _codes_with_nans(rng, M, N, K)
    sa, sb = np.float32(0.03), np.float32(1.7)
    fl.fp8la_set_gemm_variant(variant)
    try:
        C = fl.gemm(to_dev(A), to_dev(B), torch.tensor([sa], device="cuda"),
                    torch.tensor([sb], device="cuda"))
        torch.cuda.synchronize()
    finally:
        fl.fp8la_set_gemm_variant(0)
    assert fl.device_status() == 0
    r, _ = oracle.gemm_pertensor(A, B, sa, sb)
    _check(bf16_to_f64(C), r, oracle.tolerance_pertensor(A, B, sa, sb, r),
           "variant %d" % variant)


def test_blockscaled_gemm_nan_codes():
    import torch
    fl = lib()
    rng = np.random.default_rng(44)
    M, N, K = 300, 260, 96
    A, B = _codes_with_nans(rng, M, N, K)
    sa = rng.uniform(0.01, 2, (-(-M // 32), K // 32)).astype(np.float32)
    sb = rng.uniform(0.01, 2, (-(-N // 32), K // 32)).astype(np.float32)

    def dev_scales(s):
        d = torch.zeros((s.shape[0], 4), dtype=torch.float32, device="cuda")
        d[:, :s.shape[1]] = to_dev(s)
        return d[:, :s.shape[1]]

    C = fl.gemm_blockscaled_32x32(to_dev(A), to_dev(B), dev_scales(sa), dev_scales(sb))
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    r, _ = oracle.gemm_blockscaled_32x32(A, B, sa, sb)
    _check(bf16_to_f64(C), r, oracle.tolerance_blockscaled_32x32(A, B, sa, sb, r),
           "block-scaled")


@pytest.mark.parametrize("variant", [1, 2])
def test_grouped_gemm_nan_codes(variant):
    import torch
    fl = lib()
    rng = np.random.default_rng(46 + variant)
    E, N, K = 3, 260, 96
    offs = np.array([0, 140, 140, 300], np.int32)
    A = random_codes(rng, (300, K))
    B = random_codes(rng, (E, N, K))
    A[5, 10] = 0x7F            # group 0
    A[299, 0] = 0xFF           # group 2
    B[2, 7, 3] = 0x7F          # column 7 of group 2
    sa = rng.uniform(0.01, 2, E).astype(np.float32)
    sb = rng.uniform(0.01, 2, E).astype(np.float32)
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
    for e in (0, 2):
        lo, hi = offs[e], offs[e + 1]
        _check(got[lo:hi], r[lo:hi],
               oracle.tolerance_pertensor(A[lo:hi], B[e], sa[e], sb[e], r[lo:hi]),
               "variant %d group %d" % (variant, e))
