"""Pins for the oracle's scaled E4M3 GEMMs (CPU only).

Pins: the hand-worked cases in tests/golden/gemm_hand_cases.json; exact
rational brute force on tiny non-square shapes (catches transposed operands
and wrong indices); identity and permutation operands; power-of-two scales;
saturated operands; the transpose identity; PyTorch's own float8 decode plus
an fp64 matmul as a library special case; and, for the variants, reductions
to the per-tensor GEMM.  Mutants of the oracle (a transposed operand, a
dropped scale, a wrong K-block scale index) must fail these pins.
"""

import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle.e4m3 import NAN_CODE

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FINITE = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


def _codes(rng, shape):
    return rng.choice(FINITE, size=shape).astype(np.uint8)


def _dec_frac(c):
    s, e, m = (c >> 7) & 1, (c >> 3) & 15, c & 7
    v = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -v if s else v


def _rne_fraction(q):
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


def _c_float(C):
    return oracle.bf16_bits_to_float(C)


# ---------------------------------------------------------------- pin suite
def _pins_pertensor(gemm):
    """All per-tensor pins as one predicate over a gemm function."""
    try:
        with open(os.path.join(GOLDEN, "gemm_hand_cases.json")) as f:
            cases = json.load(f)["cases"]
        for c in cases:
            A = np.array([[int(v, 16) for v in row] for row in c["A"]], dtype=np.uint8)
            B = np.array([[int(v, 16) for v in row] for row in c["B"]], dtype=np.uint8)
            r, C = gemm(A, B, np.float32(c["scale_a"]), np.float32(c["scale_b"]))
            if not np.array_equal(r, np.array(c["exact"])):
                return False
            want = np.array([[int(v, 16) for v in row] for row in c["C_bf16_bits"]], dtype=np.uint16)
            if not np.array_equal(C, want):
                return False
        rng = np.random.default_rng(21)
        # brute force with exact rationals on non-square shapes
        for (M, N, K) in [(2, 3, 4), (3, 2, 5), (1, 4, 3)]:
            A, B = _codes(rng, (M, K)), _codes(rng, (N, K))
            sa, sb = np.float32(rng.uniform(0.01, 3)), np.float32(rng.uniform(0.01, 3))
            r, C = gemm(A, B, sa, sb)
            for m in range(M):
                for n in range(N):
                    q = Fraction(float(sa)) * Fraction(float(sb)) * sum(
                        _dec_frac(int(A[m, k])) * _dec_frac(int(B[n, k])) for k in range(K))
                    if _c_float(C[m:m + 1, n:n + 1])[0, 0] != float(_rne_fraction(q)):
                        return False
        # identity: A = I (0x38 = 1.0) gives C = dec(B) transposed, exactly
        N, K = 5, 7
        B = _codes(rng, (N, K))
        I = np.where(np.eye(K, dtype=bool), 0x38, 0x00).astype(np.uint8)
        r, C = gemm(I, B, 1.0, 1.0)
        if not np.array_equal(_c_float(C), oracle.decode(B).T):
            return False
        # permutation of A's rows permutes C's rows
        A = _codes(rng, (6, K))
        p = rng.permutation(6)
        _, C1 = gemm(A, B, 1.0, 1.0)
        _, C2 = gemm(A[p], B, 1.0, 1.0)
        if not np.array_equal(C1[p], C2):
            return False
        # power-of-two scale shifts exponents exactly
        r1, _ = gemm(A, B, 1.0, 1.0)
        r2, _ = gemm(A, B, np.float32(2.0 ** -5), np.float32(8.0))
        if not np.array_equal(r1 * 2.0 ** -2, r2):
            return False
        # saturated operands: 448 * 448 * K exact
        K = 3
        r, C = gemm(np.full((1, K), 0x7E, np.uint8), np.full((1, K), 0x7E, np.uint8), 1.0, 1.0)
        if r[0, 0] != 448.0 * 448.0 * K or _c_float(C)[0, 0] != 602112.0:
            return False
        # transpose: swapping the operands gives C^T
        A, B = _codes(rng, (4, 9)), _codes(rng, (3, 9))
        ra, _ = gemm(A, B, 0.5, 3.0)
        rb, _ = gemm(B, A, 3.0, 0.5)
        if not np.array_equal(ra, rb.T):
            return False
        return True
    except Exception:
        return False


def test_pertensor_pins_pass():
    assert _pins_pertensor(oracle.gemm_pertensor)


def _mut_transposed_b(A, B, sa, sb):
    return oracle.gemm_pertensor(A, B.T.copy() if B.shape[0] == B.shape[1] else B[:, ::-1], sa, sb)


def _mut_dropped_scale(A, B, sa, sb):
    return oracle.gemm_pertensor(A, B, sa, 1.0)


def _mut_fp32_rounding(A, B, sa, sb):
    r, _ = oracle.gemm_pertensor(A, B, sa, sb)
    return r, oracle.bf16_rne(r.astype(np.float32).astype(np.float64))


def _mut_wrong_sign(A, B, sa, sb):
    return oracle.gemm_pertensor(A & 0x7F, B, sa, sb)


@pytest.mark.parametrize("mutant", [_mut_transposed_b, _mut_dropped_scale,
                                    _mut_fp32_rounding, _mut_wrong_sign])
def test_planted_gemm_mistakes_are_caught(mutant):
    assert not _pins_pertensor(mutant)


def test_matches_torch_float8_decode_and_matmul():
    rng = np.random.default_rng(22)
    A, B = _codes(rng, (37, 64)), _codes(rng, (29, 64))
    Ad = torch.from_numpy(A).view(torch.float8_e4m3fn).to(torch.float64)
    Bd = torch.from_numpy(B).view(torch.float8_e4m3fn).to(torch.float64)
    ref = (Ad @ Bd.T * (0.25 * 0.125)).numpy()
    r, _ = oracle.gemm_pertensor(A, B, 0.25, 0.125)
    assert np.array_equal(r, ref)


def test_row_col_sampling_matches_full():
    rng = np.random.default_rng(23)
    A, B = _codes(rng, (40, 48)), _codes(rng, (33, 48))
    r, C = oracle.gemm_pertensor(A, B, 0.3, 0.7)
    rows, cols = np.array([0, 5, 39]), np.array([32, 1])
    rs, Cs = oracle.gemm_pertensor(A, B, 0.3, 0.7, rows=rows, cols=cols)
    assert np.array_equal(C[np.ix_(rows, cols)], Cs)


# ------------------------------------------------------------ block-scaled
def _pins_block(gemm_block):
    try:
        rng = np.random.default_rng(31)
        M, N, K = 70, 45, 100
        A, B = _codes(rng, (M, K)), _codes(rng, (N, K))
        ta, tb, tk = -(-M // 32), -(-N // 32), -(-K // 32)
        # all tile scales equal -> per-tensor result, bit for bit
        sa = np.full((ta, tk), 0.375, np.float32)
        sb = np.full((tb, tk), 1.25, np.float32)
        r1, C1 = gemm_block(A, B, sa, sb)
        r0, C0 = oracle.gemm_pertensor(A, B, 0.375, 1.25)
        if not (np.array_equal(C1, C0) and np.allclose(r1, r0, rtol=1e-15, atol=0)):
            return False
        # one-hot tile scale isolates one K block
        for kb in range(tk):
            sa = np.zeros((ta, tk), np.float32)
            sb = np.ones((tb, tk), np.float32)
            sa[:, kb] = 2.0
            r, _ = gemm_block(A, B, sa, sb)
            ks = slice(32 * kb, min(32 * kb + 32, K))
            rk, _ = oracle.gemm_pertensor(A[:, ks], B[:, ks], 2.0, 1.0)
            if not np.array_equal(r, rk):
                return False
        # row-tile scale only scales its 32 rows
        sa = np.ones((ta, tk), np.float32)
        sa[1, :] = 4.0
        sb = np.ones((tb, tk), np.float32)
        r, _ = gemm_block(A, B, sa, sb)
        rp, _ = oracle.gemm_pertensor(A, B, 1.0, 1.0)
        scale_rows = np.ones(M)
        scale_rows[32:64] = 4.0
        if not np.array_equal(r, rp * scale_rows[:, None]):
            return False
        # exact rational brute force on a small ragged case
        M, N, K = 3, 2, 40
        A, B = _codes(rng, (M, K)), _codes(rng, (N, K))
        sa = rng.uniform(0.1, 2, (1, 2)).astype(np.float32)
        sb = rng.uniform(0.1, 2, (1, 2)).astype(np.float32)
        _, C = gemm_block(A, B, sa, sb)
        for m in range(M):
            for n in range(N):
                q = Fraction(0)
                for kb in range(2):
                    s = Fraction(float(sa[0, kb])) * Fraction(float(sb[0, kb]))
                    q += s * sum(_dec_frac(int(A[m, k])) * _dec_frac(int(B[n, k]))
                                 for k in range(32 * kb, min(32 * kb + 32, K)))
                if _c_float(C[m:m + 1, n:n + 1])[0, 0] != float(_rne_fraction(q)):
                    return False
        return True
    except Exception:
        return False


def test_block_pins_pass():
    assert _pins_block(oracle.gemm_blockscaled_32x32)


def _mut_block_index(A, B, sa, sb):
    # uses the K-block index of the scale grid in reverse
    return oracle.gemm_blockscaled_32x32(A, B, sa[:, ::-1].copy(), sb, )


def _mut_block_size_64(A, B, sa, sb):
    sa2 = np.repeat(sa[:, ::2], 2, axis=1)[:, :sa.shape[1]].copy()
    return oracle.gemm_blockscaled_32x32(A, B, sa2, sb)


@pytest.mark.parametrize("mutant", [_mut_block_index, _mut_block_size_64])
def test_planted_block_mistakes_are_caught(mutant):
    assert not _pins_block(mutant)


# ------------------------------------------------------------------ grouped
def test_grouped_equals_separate_calls_and_skips_empty_groups():
    rng = np.random.default_rng(41)
    E, N, K = 5, 24, 48
    counts = np.array([7, 0, 33, 0, 1])
    off = np.concatenate([[0], np.cumsum(counts)])
    A = _codes(rng, (off[-1], K))
    B = _codes(rng, (E, N, K))
    sa = rng.uniform(0.1, 2, E).astype(np.float32)
    sb = rng.uniform(0.1, 2, E).astype(np.float32)
    r, C = oracle.gemm_grouped(A, off, B, sa, sb)
    assert C.shape == (off[-1], N)
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        re, Ce = oracle.gemm_pertensor(A[lo:hi], B[e], sa[e], sb[e])
        assert np.array_equal(C[lo:hi], Ce)
    # all-empty
    r, C = oracle.gemm_grouped(A[:0], np.zeros(E + 1, np.int64), B, sa, sb)
    assert C.shape == (0, N)


def test_nan_code_constant():
    assert NAN_CODE == 0x7F


def test_bound_covers_one_rounding():
    """The bound admits bf16(r) itself and one fp32-level perturbation."""
    rng = np.random.default_rng(51)
    A, B = _codes(rng, (16, 256)), _codes(rng, (16, 256))
    r, C = oracle.gemm_pertensor(A, B, 0.01, 0.02)
    maxa = np.abs(oracle.decode(A)).max()
    maxb = np.abs(oracle.decode(B)).max()
    bnd = oracle.bound_pertensor(r, 256, 0.01, 0.02, maxa, maxb)
    assert np.all(np.abs(_c_float(C) - r) <= bnd)
