"""Scaled E4M3 GEMMs: per-tensor, 32x32 block-scaled and grouped (MoE).

Operand layout used throughout: A is [M][K] (row m holds A[m, 0..K-1]); B is
stored K-major as [N][K] (row n holds the K values of column n of the K x N
matrix), so the product is C[m, n] = sum_k A[m, k] * B[n, k].

Exactness of the sum.  Every E4M3 value is (integer < 16) * 2^j with
j >= -9, so every product dec(a) * dec(b) is a multiple of 2^-18 with at most
8 significant bits, and |product| <= 448^2 < 2^18.  A sum of K such products
is a multiple of 2^-18 of magnitude below K * 2^18; for K < 2^17 it is below
2^35 = 2^53 * 2^-18, so every partial sum, in any order and with or without
fused multiply-adds, is exactly representable in fp64.  An fp64 matrix
product (a library primitive) therefore returns the exact integer-lattice
sum S, and the only rounding in r = (sa * sb) * S is the final fp64
multiply (sa * sb itself is exact: two 24-bit significands).

Scales are applied once to the finished sum (per-tensor) or once per 32-wide
K block (block-scaled).  [P1] (scale paragraph, "此内核借鉴 CUTLASS") writes
``acc = acc * scale_a * scale_b``; applied once to the full FP32 sum, per
tensor, this is the same mathematics.

Each function returns (r, C): r the fp64 value before the output rounding,
and C its bf16 RNE rounding as uint16 bit patterns.
"""

import numpy as np

from . import e4m3, e5m2
from .e4m3 import decode
from .bf16 import bf16_rne

DECODERS = {"e4m3": e4m3.decode, "e5m2": e5m2.decode}

KMAX_EXACT = 1 << 17


def _rows_cols(M, N, rows, cols):
    rows = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    cols = np.arange(N) if cols is None else np.asarray(cols, dtype=np.int64)
    return rows, cols


def gemm_pertensor(A, B, scale_a, scale_b, rows=None, cols=None,
                   a_fmt="e4m3", b_fmt="e4m3"):
    """C[m, n] = bf16_RNE(sa * sb * sum_k dec(A[m, k]) * dec(B[n, k])).

    FP32 accumulation is the kernel's choice ([P1], parameter list "累加器
    FP32"); the oracle sums exactly instead (see the module docstring).
    ``rows``/``cols`` restrict the result to C[rows][:, cols].  a_fmt,
    b_fmt select each operand's FP8 format ("e4m3" or "e5m2").  With an E5M2
    operand the products span more than 53 bits, so the fp64 sum is exact
    only up to a relative rounding of 2^-53 per addition -- 2^-31 of the
    accumulation term of the error bound.
    """
    A = np.asarray(A, dtype=np.uint8)
    B = np.asarray(B, dtype=np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("A and B disagree on K")
    if K >= KMAX_EXACT:
        raise ValueError("K too large for an exact fp64 sum")
    rows, cols = _rows_cols(M, N, rows, cols)
    Ad = DECODERS[a_fmt](A[rows])              # [m][k], fp64
    Bd = DECODERS[b_fmt](B[cols])              # [n][k], fp64
    S = Ad @ Bd.T                              # exact (E4M3 x E4M3)
    r = (np.float64(np.float32(scale_a)) * np.float64(np.float32(scale_b))) * S
    return r, bf16_rne(r)


def gemm_blockscaled_32x32(A, B, sa, sb, rows=None, cols=None):
    """C[m, n] = bf16_RNE(sum_kb sa[m//32, kb] * sb[n//32, kb] * S_kb[m, n]).

    S_kb is the exact sum over the kb-th 32-wide K block (the last block cut
    short at K).  sa is [ceil(M/32)][ceil(K/32)] and sb is
    [ceil(N/32)][ceil(K/32)], one fp32 scale per 32x32 tile of each operand
    ([P3], implementation paragraph: "缩放粒度为 32x32 块（microscaling）").
    The per-block partial sums are weighted by their own scales and added in
    fp64; that is the promotion of each K block's partial into the
    accumulator that [P3] (warp specialisation paragraph) assigns to a
    CUDA-core warp.
    """
    A = np.asarray(A, dtype=np.uint8)
    B = np.asarray(B, dtype=np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("A and B disagree on K")
    nkb = -(-K // 32)
    sa = np.asarray(sa, dtype=np.float32)
    sb = np.asarray(sb, dtype=np.float32)
    if sa.shape != (-(-M // 32), nkb) or sb.shape != (-(-N // 32), nkb):
        raise ValueError("scale grids have the wrong shape")
    rows, cols = _rows_cols(M, N, rows, cols)
    Ad = decode(A[rows])
    Bd = decode(B[cols])
    r = np.zeros((rows.size, cols.size), dtype=np.float64)
    for kb in range(nkb):
        ks = slice(32 * kb, min(32 * kb + 32, K))
        S_kb = Ad[:, ks] @ Bd[:, ks].T                     # exact
        w = (sa[rows // 32, kb].astype(np.float64)[:, None]
             * sb[cols // 32, kb].astype(np.float64)[None, :])  # exact
        r += w * S_kb
    return r, bf16_rne(r)


def gemm_grouped(A, m_offsets, B, scale_a, scale_b, cols=None):
    """Grouped per-tensor GEMM over E groups (MoE experts).

    Group e owns rows m_offsets[e] .. m_offsets[e+1]-1 of the concatenated
    A [sum M_e][K] and of C; its weights are B[e] ([N][K], K-major) and its
    scales scale_a[e], scale_b[e].  C rows of group e are
    gemm_pertensor(A[rows of e], B[e], scale_a[e], scale_b[e]).  Groups with
    M_e = 0 produce nothing ([P3], implementation paragraph: "对于 MoE 场景，
    扩展为分组 GEMM").  Rows at or past m_offsets[E] are not produced.

    Returns (r, C) over rows 0 .. m_offsets[E]-1.
    """
    A = np.asarray(A, dtype=np.uint8)
    B = np.asarray(B, dtype=np.uint8)
    off = np.asarray(m_offsets, dtype=np.int64)
    E = off.size - 1
    if B.ndim != 3 or B.shape[0] != E:
        raise ValueError("B must be [E][N][K]")
    if np.any(np.diff(off) < 0) or off[0] != 0:
        raise ValueError("m_offsets must start at 0 and be non-decreasing")
    N = B.shape[1]
    ncols = N if cols is None else len(cols)
    Mtot = int(off[-1])
    r = np.zeros((Mtot, ncols), dtype=np.float64)
    C = np.zeros((Mtot, ncols), dtype=np.uint16)
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        r_e, C_e = gemm_pertensor(A[lo:hi], B[e], scale_a[e], scale_b[e],
                                  cols=cols)
        r[lo:hi] = r_e
        C[lo:hi] = C_e
    return r, C


def max_abs_decoded(codes, fmt="e4m3"):
    """max over the codes of |dec(code)|, NaN codes left out (0 if none).

    This is the "max|a|" (or "max|b|") of the error bound below: a maximum
    over the DECODED operand values, not over the raw byte codes.
    """
    d = np.abs(DECODERS[fmt](np.asarray(codes, dtype=np.uint8)))
    d = d[~np.isnan(d)]
    return float(d.max()) if d.size else 0.0


def max_abs_tile_scaled_32x32(codes, s):
    """max over (m, k) of |s[m//32, k//32] * dec(codes[m, k])| (NaN codes left out).

    The block-scaled form of sa * max|a| in the error bound: each decoded
    value is weighted by the scale of the 32x32 tile that holds it before the
    maximum is taken.  Every product is exact in fp64 (a 24-bit scale times a
    decoded value of at most 4 significant bits).
    """
    codes = np.asarray(codes, dtype=np.uint8)
    s = np.asarray(s, dtype=np.float32).astype(np.float64)
    M, K = codes.shape
    best = 0.0
    for r0 in range(0, M, 2048):                      # bounded memory
        blk = np.abs(decode(codes[r0:r0 + 2048]))
        rows = np.arange(r0, r0 + blk.shape[0]) // 32
        cols = np.arange(K) // 32
        w = np.abs(s[rows][:, cols]) * blk
        w = w[~np.isnan(w)]
        if w.size:
            best = max(best, float(w.max()))
    return best


def bound_pertensor(r, K, scale_a, scale_b, max_a, max_b):
    """Allowed |C_gpu - C_ref| per element for a per-tensor GEMM.

    2^-8 * |C_ref| + 2^-22 * K * sa * sb * max|a| * max|b|, with a, b the
    decoded E4M3 operand values (``max_abs_decoded``) and C_ref the exact
    product r.  The first term is one bf16 rounding (unit roundoff 2^-8); the
    second covers an FP32 accumulation over K terms (4x the fp32 unit
    roundoff 2^-24 per term, relative to the largest possible product).
    """
    return (2.0 ** -8) * np.abs(r) + (2.0 ** -22) * K * (
        float(np.float32(scale_a)) * float(np.float32(scale_b))
        * float(max_a) * float(max_b))


def bound_blockscaled_32x32(r, K, max_sa_a, max_sb_b):
    """The block-scaled form of ``bound_pertensor``.

    sa * max|a| is replaced by max over (m, k) of |sa[m//32, k//32] * dec(a)|
    and likewise for B (``max_abs_tile_scaled_32x32``); the caller passes
    those two maxima.
    """
    return (2.0 ** -8) * np.abs(r) + (2.0 ** -22) * K * float(max_sa_a) * float(max_sb_b)


def tolerance_pertensor(A, B, scale_a, scale_b, r, a_fmt="e4m3", b_fmt="e4m3"):
    """The per-element bound for C = gemm_pertensor(A, B, scale_a, scale_b).

    ``r`` is the oracle's exact product (for the whole matrix or any subset
    of its elements); the maxima run over ALL of A and B.
    """
    K = np.asarray(A).shape[1]
    return bound_pertensor(r, K, scale_a, scale_b,
                           max_abs_decoded(A, a_fmt), max_abs_decoded(B, b_fmt))


def tolerance_blockscaled_32x32(A, B, sa, sb, r):
    """The per-element bound for C = gemm_blockscaled_32x32(A, B, sa, sb)."""
    K = np.asarray(A).shape[1]
    return bound_blockscaled_32x32(r, K, max_abs_tile_scaled_32x32(A, sa),
                                   max_abs_tile_scaled_32x32(B, sb))
