"""Shared helpers for the GPU parity tests (comparison against the oracle)."""

import numpy as np

import oracle

FINITE_CODES = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


def lib():
    import precision_linear_algebra_gb300 as fl
    from precision_linear_algebra_gb300 import build
    build.build()
    fl.load()
    return fl


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_to_f64(t):
    """torch bf16 tensor -> numpy fp64 (exact)."""
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32).__lshift__(16).view(np.float32).astype(np.float64)


def bf16_bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def random_codes(rng, shape):
    return rng.choice(FINITE_CODES, size=shape).astype(np.uint8)


def assert_within_bound(C_gpu, r, bound, what=""):
    """Assert |C_gpu - r| <= bound elementwise and that C_gpu is finite.

    C_gpu, r, bound: numpy fp64 arrays of one shape (r the oracle's exact
    product, bound from oracle.tolerance_*).  NaN or Inf in C_gpu fails.
    """
    assert np.all(np.isfinite(C_gpu)), what + ": non-finite output"
    err = np.abs(C_gpu - r)
    bad = ~(err <= bound)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(
            "%s: %d/%d outside bound; first at %s: got %r want %r (bound %r)"
            % (what, bad.sum(), bad.size, i, C_gpu[i], r[i], bound[i]))


def check_pertensor(C_gpu, A, B, sa, sb, rows=None, cols=None, what=""):
    """Assert the bound |C_gpu - r| <= 2^-8|r| + 2^-22 K sa sb max|a| max|b|.

    A, B: oracle-side codes; C_gpu: numpy fp64 values at (rows, cols) (or the
    whole matrix).  Returns the fraction of outputs equal to bf16_RNE(r).
    """
    K = A.shape[1]
    r, Cref = oracle.gemm_pertensor(A, B, sa, sb, rows=rows, cols=cols)
    if K == 0:
        assert np.all(C_gpu == 0), what
        return 1.0
    assert_within_bound(C_gpu, r, oracle.tolerance_pertensor(A, B, sa, sb, r), what)
    return float(np.mean(C_gpu == oracle.bf16_bits_to_float(Cref)))
