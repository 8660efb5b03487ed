"""GPU parity on seeded random shapes (a shape fuzzer).

Every GEMM kernel runs on ragged M, N, K drawn at random, and every output is
checked against the oracle within its bound:

    |C_gpu - C_ref| <= 2^-8 |C_ref| + 2^-22 K max|scaled a| max|scaled b|

Guard columns past N and guard rows past M (past the last group for the
grouped GEMM) must come back untouched.  The quantisers run on random ragged
shapes with padded row strides and must match the oracle bit for bit.
Shapes, codes and scales come from fixed seeds, so a failure reproduces.
FP8LA_FUZZ_MULT=n runs n times as many cases of each kind; the first ones
are the default run's.
"""

import os

import numpy as np
import pytest

import oracle
from _helpers import assert_within_bound, bf16_to_f64, lib, random_codes, to_dev

pytestmark = pytest.mark.gpu

_MULT = max(1, int(os.environ.get("FP8LA_FUZZ_MULT", "1")))

SENTINEL = -7.0


def _shapes(seed, n, hi=700):
    rng = np.random.default_rng(seed)
    return [tuple(int(v) for v in rng.integers(1, hi, 3)) for _ in range(n)]


def _dev_codes(codes):
    """Codes on the device with rows padded to a multiple of 16 bytes (the
    GEMMs read operands by TMA); returns the [rows][K] view."""
    import torch
    rows, K = codes.shape
    kp = max(16, (K + 15) // 16 * 16)
    d = torch.zeros((rows, kp), dtype=torch.uint8, device="cuda")
    d[:, :K] = to_dev(codes)
    return d[:, :K]


def _guarded_c(rows, N, aligned, extra_rows=5):
    """C with guard rows and columns around the [rows][N] view; `aligned`
    makes the row stride a multiple of 8 (16 bytes), so that the GEMMs may
    store whole blocks by TMA, else it is not (row-by-row stores)."""
    import torch
    extra_cols = 8 + (-N) % 8 if aligned else 8 + (1 if (N + 8) % 8 == 0 else 0)
    full = torch.full((rows + extra_rows, N + extra_cols), SENTINEL,
                      dtype=torch.bfloat16, device="cuda")
    return full, full[:rows, :N]


def _guards_untouched(full, rows, N):
    f = bf16_to_f64(full)
    return np.all(f[rows:, :] == SENTINEL) and np.all(f[:, N:] == SENTINEL)


@pytest.mark.parametrize("case", range(40 * _MULT))
def test_pertensor_gemm_random_shapes(case):
    import torch
    fl = lib()
    M, N, K = _shapes(101, 40 * _MULT)[case]
    variant = [0, 1, 2, 3, 4][case % 5]
    rng = np.random.default_rng(1000 + case)
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa, sb = (np.float32(v) for v in rng.uniform(1e-3, 2.0, 2))
    full, C = _guarded_c(M, N, aligned=case % 3 != 2)
    fl.fp8la_set_gemm_variant(variant)
    try:
        fl.gemm(_dev_codes(A), _dev_codes(B),
                torch.tensor([sa], dtype=torch.float32, device="cuda"),
                torch.tensor([sb], dtype=torch.float32, device="cuda"), C=C)
        torch.cuda.synchronize()
    finally:
        fl.fp8la_set_gemm_variant(0)
    assert fl.device_status() == 0
    what = "%dx%dx%d variant %d" % (M, N, K, variant)
    assert _guards_untouched(full, M, N), what + ": write outside C"
    r, _ = oracle.gemm_pertensor(A, B, sa, sb)
    assert_within_bound(bf16_to_f64(C.contiguous()), r,
                        oracle.tolerance_pertensor(A, B, sa, sb, r), what)


@pytest.mark.parametrize("case", range(30 * _MULT))
def test_blockscaled_gemm_random_shapes(case):
    import torch
    fl = lib()
    M, N, K = _shapes(202, 30 * _MULT)[case]
    rng = np.random.default_rng(2000 + case)
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    nkb = -(-K // 32)
    sa = rng.uniform(1e-3, 2.0, (-(-M // 32), nkb)).astype(np.float32)
    sb = rng.uniform(1e-3, 2.0, (-(-N // 32), nkb)).astype(np.float32)

    def dev_scales(s):
        rows, c = s.shape
        d = torch.full((rows, (c + 3) // 4 * 4), float("nan"), dtype=torch.float32,
                       device="cuda")
        d[:, :c] = to_dev(s)
        return d[:, :c]

    full, C = _guarded_c(M, N, aligned=case % 3 != 2)
    fl.gemm_blockscaled_32x32(_dev_codes(A), _dev_codes(B), dev_scales(sa), dev_scales(sb),
                              C=C)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    what = "%dx%dx%d" % (M, N, K)
    assert _guards_untouched(full, M, N), what + ": write outside C"
    r, _ = oracle.gemm_blockscaled_32x32(A, B, sa, sb)
    assert_within_bound(bf16_to_f64(C.contiguous()), r,
                        oracle.tolerance_blockscaled_32x32(A, B, sa, sb, r), what)


@pytest.mark.parametrize("case", range(24 * _MULT))
def test_grouped_gemm_random_shapes(case):
    import torch
    fl = lib()
    rng = np.random.default_rng(3000 + case)
    E = int(rng.integers(1, 10))
    counts = rng.integers(0, 400, E) * (rng.random(E) > 0.25)   # some groups empty
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(offs[-1])
    N = int(rng.integers(1, 600))
    K = int(rng.integers(1, 600))
    A = random_codes(rng, (max(rows, 1), K))[:rows]
    B = random_codes(rng, (E, N, K))
    sa = rng.uniform(0.01, 2, E).astype(np.float32)
    sb = rng.uniform(0.01, 2, E).astype(np.float32)
    cap = rows + 37
    kp = max(16, (K + 15) // 16 * 16)
    dA = torch.zeros((cap, kp), dtype=torch.uint8, device="cuda")
    dA[:rows, :K] = to_dev(A)
    dB = torch.zeros((E, N, kp), dtype=torch.uint8, device="cuda")
    dB[:, :, :K] = to_dev(B)
    ldc = N + 8 + ((-N) % 8 if case % 2 == 0 else (1 if (N + 8) % 8 == 0 else 0))
    full = torch.full((cap, ldc), SENTINEL, dtype=torch.bfloat16, device="cuda")
    # device copies held in names: a temporary's memory could be reused by
    # the next allocation before the kernel reads it
    d_off, d_sa, d_sb = to_dev(offs), to_dev(sa), to_dev(sb)
    variant = 1 + case % 2
    fl.fp8la_set_gemm_variant(variant)
    try:
        fl.fp8_grouped_gemm(E, d_off.data_ptr(), cap, dA.data_ptr(), kp, dB.data_ptr(),
                            kp, N * kp, full.data_ptr(), ldc, N, K,
                            d_sa.data_ptr(), d_sb.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
    finally:
        fl.fp8la_set_gemm_variant(0)
    assert fl.device_status() == 0
    what = "E %d rows %d N %d K %d variant %d" % (E, rows, N, K, variant)
    got = bf16_to_f64(full)
    assert np.all(got[rows:, :] == SENTINEL), what + ": rows past the last group written"
    assert np.all(got[:, N:] == SENTINEL), what + ": columns past N written"
    r, _ = oracle.gemm_grouped(A, offs, B, sa, sb)
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi > lo:
            assert_within_bound(got[lo:hi, :N], r[lo:hi],
                                oracle.tolerance_pertensor(A[lo:hi], B[e], sa[e], sb[e],
                                                           r[lo:hi]),
                                what + " group %d" % e)


@pytest.mark.parametrize("case", range(30 * _MULT))
def test_quantisers_random_shapes(case):
    """Per-tensor (E4M3 and E5M2) and 32x32 block quantisation of random
    ragged shapes with padded row strides, bit for bit."""
    import torch
    fl = lib()
    rng = np.random.default_rng(4000 + case)
    rows, cols = (int(v) for v in rng.integers(1, 1500, 2))
    x = (rng.standard_normal((rows, cols)) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
    pad = int(rng.integers(0, 9))
    dfull = torch.zeros((rows, cols + pad), dtype=torch.float32, device="cuda")
    dfull[:, :cols] = to_dev(x)
    dx = dfull[:, :cols]
    fmt = ("e4m3", "e5m2")[case % 2]
    q, amax, scale = fl.quantize_pertensor(dx, fmt=fmt)
    rq, ramax, rscale = oracle.quantize_pertensor(x, fmt=fmt)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    assert np.array_equal(q.cpu().numpy(), rq), (rows, cols, fmt)
    assert amax.item() == ramax and scale.item() == rscale
    # 16-byte loads when cols and the row stride allow, scalar loads otherwise
    qb, sb = fl.quantize_blockwise_32x32(dx)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    rqb, rsb = oracle.quantize_blockwise_32x32(x)
    assert np.array_equal(qb.cpu().numpy(), rqb), (rows, cols, pad)
    assert np.array_equal(sb.cpu().numpy(), rsb), (rows, cols, pad)


@pytest.mark.parametrize("case", range(16 * _MULT))
def test_grouped_quantiser_random_shapes(case):
    """Grouped per-tensor quantisation of random ragged groups (some empty)
    with padded strides and guard rows past the last group, bit for bit."""
    import torch
    fl = lib()
    rng = np.random.default_rng(5000 + case)
    E = int(rng.integers(1, 17))
    counts = rng.integers(0, 200, E) * (rng.random(E) > 0.3)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows, cols = int(offs[-1]), int(rng.integers(1, 900))
    cap = rows + int(rng.integers(0, 20))
    pad = int(rng.integers(0, 9))
    x = (rng.standard_normal((rows, cols)) * 10.0 ** rng.uniform(-4, 4)).astype(np.float32)
    dfull = torch.zeros((cap, cols + pad), dtype=torch.float32, device="cuda")
    dfull[:rows, :cols] = to_dev(x)
    qfull = torch.full((cap, cols + pad), 0xA5, dtype=torch.uint8, device="cuda")
    d_off = to_dev(offs)
    q, amax, scale = fl.quantize_pertensor_grouped(dfull[:, :cols], d_off, q=qfull[:, :cols])
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    rq, ramax, rscale = oracle.quantize_pertensor_grouped(x, offs)
    got = qfull.cpu().numpy()
    assert np.array_equal(got[:rows, :cols], rq), (E, rows, cols, pad)
    assert np.array_equal(amax.cpu().numpy(), ramax) and np.array_equal(scale.cpu().numpy(), rscale)
    assert np.all(got[rows:] == 0xA5) and np.all(got[:, cols:] == 0xA5)


@pytest.mark.parametrize("case", range(20 * _MULT))
def test_quantisers_special_values_random(case):
    """Per-tensor (E4M3, E5M2), delayed and block quantisers on random
    ragged shapes with magnitudes spread over 40 binades and special values
    (+-Inf, NaN, +-0, fp32 subnormals, the fp32 maximum) sprinkled in, bit
    for bit."""
    import torch
    fl = lib()
    rng = np.random.default_rng(6000 + case)
    rows, cols = (int(v) for v in rng.integers(1, 400, 2))
    x = (rng.standard_normal((rows, cols))
         * 2.0 ** rng.uniform(-20, 20, (rows, cols))).astype(np.float32)
    specials = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, 1e-41, -3e-39,
                         3.4e38, -3.4e38], np.float32)
    n_sp = int(rng.integers(0, 6))
    if n_sp:
        idx = rng.integers(0, x.size, n_sp)
        x.reshape(-1)[idx] = rng.choice(specials, n_sp)
    dx = to_dev(x)
    fmt = ("e4m3", "e5m2")[case % 2]
    q, amax, scale = fl.quantize_pertensor(dx, fmt=fmt)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    rq, ramax, rscale = oracle.quantize_pertensor(x, fmt=fmt)
    assert np.array_equal(q.cpu().numpy(), rq), (rows, cols, fmt)
    assert np.float32(amax.item()).tobytes() == np.float32(ramax).tobytes()
    assert np.float32(scale.item()).tobytes() == np.float32(rscale).tobytes()
    prev = float(rng.choice([ramax, 1.0, 1e-30, np.inf, 448.0]))
    dprev = torch.tensor([prev], dtype=torch.float32, device="cuda")
    q2, amax2, scale2 = fl.quantize_pertensor_delayed(dx, dprev, fmt=fmt)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    rq2, ramax2, rscale2 = oracle.quantize_pertensor_delayed(x, prev, fmt)
    assert np.array_equal(q2.cpu().numpy(), rq2), (rows, cols, fmt, prev)
    assert np.float32(amax2.item()).tobytes() == np.float32(ramax2).tobytes()
    assert np.float32(scale2.item()).tobytes() == np.float32(rscale2).tobytes()
    qb, sbk = fl.quantize_blockwise_32x32(dx)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    rqb, rsb = oracle.quantize_blockwise_32x32(x)
    assert np.array_equal(qb.cpu().numpy(), rqb), (rows, cols)
    assert np.array_equal(sbk.cpu().numpy().view(np.uint32), rsb.view(np.uint32))


@pytest.mark.parametrize("case", range(20 * _MULT))
def test_gemms_wide_scale_ranges(case):
    """Per-tensor GEMM with scale pairs whose product spans 1e-25 .. 1e25 and
    block-scaled GEMM with tile scales spread over 1e-6 .. 1e6, random ragged
    shapes; every output within the bound."""
    import torch
    fl = lib()
    rng = np.random.default_rng(7000 + case)
    M, N, K = (int(v) for v in rng.integers(1, 500, 3))
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    e = rng.uniform(-25, 25)
    f = rng.uniform(0, 1)
    sa, sb = np.float32(10.0 ** (e * f)), np.float32(10.0 ** (e * (1 - f)))
    variant = [0, 1, 2, 3, 4][case % 5]
    fl.fp8la_set_gemm_variant(variant)
    try:
        C = fl.gemm(_dev_codes(A), _dev_codes(B), torch.tensor([sa], device="cuda"),
                    torch.tensor([sb], device="cuda"))
        torch.cuda.synchronize()
    finally:
        fl.fp8la_set_gemm_variant(0)
    assert fl.device_status() == 0
    what = "%dx%dx%d sa %g sb %g variant %d" % (M, N, K, sa, sb, variant)
    r, _ = oracle.gemm_pertensor(A, B, sa, sb)
    assert_within_bound(bf16_to_f64(C), r, oracle.tolerance_pertensor(A, B, sa, sb, r), what)
    nkb = -(-K // 32)
    ta = (10.0 ** rng.uniform(-6, 6, (-(-M // 32), nkb))).astype(np.float32)
    tb = (10.0 ** rng.uniform(-6, 6, (-(-N // 32), nkb))).astype(np.float32)

    def dev_scales(s):
        d = torch.zeros((s.shape[0], (s.shape[1] + 3) // 4 * 4), dtype=torch.float32,
                        device="cuda")
        d[:, :s.shape[1]] = to_dev(s)
        return d[:, :s.shape[1]]

    C2 = fl.gemm_blockscaled_32x32(_dev_codes(A), _dev_codes(B), dev_scales(ta), dev_scales(tb))
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    r2, _ = oracle.gemm_blockscaled_32x32(A, B, ta, tb)
    assert_within_bound(bf16_to_f64(C2), r2,
                        oracle.tolerance_blockscaled_32x32(A, B, ta, tb, r2),
                        "block-scaled %dx%dx%d" % (M, N, K))
