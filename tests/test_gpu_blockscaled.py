"""GPU parity: 32x32 block-scaled E4M3 GEMM against the oracle, within

    |C_gpu - C_ref| <= 2^-8 |C_ref| + 2^-22 K max|sa*a| max|sb*b|

elementwise (C_ref the oracle's product before BF16 rounding; max|sa*a| the
largest |tile scale x decoded code| of A, likewise for B)."""

import numpy as np
import pytest

import oracle
from _helpers import (assert_within_bound, bf16_to_f64, check_pertensor, lib,
                      random_codes, to_dev)
from precision_linear_algebra_gb300 import workloads

pytestmark = pytest.mark.gpu


def check_block(C_gpu, A, B, sa, sb, rows=None, cols=None, what="", maxes=None):
    """Assert the block-scaled bound; maxes = (max|sa*a|, max|sb*b|) when the
    caller has them already (full-size operands), else computed here."""
    K = A.shape[1]
    r, Cref = oracle.gemm_blockscaled_32x32(A, B, sa, sb, rows=rows, cols=cols)
    if maxes is None:
        bound = oracle.tolerance_blockscaled_32x32(A, B, sa, sb, r)
    else:
        bound = oracle.bound_blockscaled_32x32(r, K, *maxes)
    assert_within_bound(C_gpu, r, bound, what)
    return float(np.mean(C_gpu == oracle.bf16_bits_to_float(Cref)))


def _run(fl, A, B, sa, sb, ldc_pad=0):
    import torch
    M, K = A.shape
    N = B.shape[0]
    kp = max(16, (K + 15) // 16 * 16)
    dA = torch.zeros((M, kp), dtype=torch.uint8, device="cuda")
    dB = torch.zeros((N, kp), dtype=torch.uint8, device="cuda")
    dA[:, :K] = to_dev(A)
    dB[:, :K] = to_dev(B)
    Cs = torch.full((M, N + ldc_pad), 5.0, dtype=torch.bfloat16, device="cuda")
    C = Cs[:, :N]
    fl.gemm_blockscaled_32x32(dA[:, :K], dB[:, :K], _dev_scales(sa), _dev_scales(sb), C=C)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    if ldc_pad:
        assert torch.all(Cs[:, N:] == 5.0)
    return bf16_to_f64(C.contiguous())


def _dev_scales(s):
    """Scale grid on the device with its leading dimension padded to a
    multiple of 4 floats (the GEMM reads it by TMA)."""
    import torch
    r, c = s.shape
    d = torch.full((r, (c + 3) // 4 * 4), float("nan"), dtype=torch.float32, device="cuda")
    d[:, :c] = to_dev(s)
    return d[:, :c]


def _scales(rng, rows, K):
    return rng.uniform(1e-3, 2.0, (-(-rows // 32), -(-K // 32))).astype(np.float32)


@pytest.mark.parametrize("M,N,K", [
    (128, 128, 128), (128, 128, 32), (128, 128, 48), (256, 384, 512),
    (300, 200, 100), (1, 1, 16), (640, 256, 1024), (129, 130, 272),
])
def test_random_codes_random_scales(M, N, K):
    fl = lib()
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa, sb = _scales(rng, M, K), _scales(rng, N, K)
    got = _run(fl, A, B, sa, sb, ldc_pad=8 if N % 8 == 0 else 0)
    frac = check_block(got, A, B, sa, sb, what="%dx%dx%d" % (M, N, K))
    assert frac > 0.98


def test_many_tiles_per_cta_all_outputs():
    """About two 128 x 64 tiles per persistent CTA and a ragged last K stage
    (K = 320: 10 scale blocks, 2.5 stages), every output checked: a scale
    paired with the wrong K block after a tile change would show here."""
    fl = lib()
    M, N, K = 1536, 1600, 320
    rng = np.random.default_rng(77)
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa, sb = _scales(rng, M, K), _scales(rng, N, K)
    got = _run(fl, A, B, sa, sb)
    frac = check_block(got, A, B, sa, sb, what="many tiles")
    assert frac > 0.98


def test_tile_pairs_and_ring_laps_all_outputs():
    """Three 128 x 128 output tiles per persistent CTA (six of 128 x 64) and
    K = 1344 (42 scale blocks, 10.5 stages of 128, so every ring slot is
    refilled several times per tile), every output checked.  Scales read
    from a ring slot after its next fill had landed (a stage's scales
    replaced by those of a later stage) showed only after a CTA's first
    tiles.  That race depended on timing (one call in three failed), so
    three calls are checked."""
    fl = lib()
    M, N, K = 1024, 7296, 1344
    rng = np.random.default_rng(78)
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa, sb = _scales(rng, M, K), _scales(rng, N, K)
    r, Cref = oracle.gemm_blockscaled_32x32(A, B, sa, sb)
    bound = oracle.tolerance_blockscaled_32x32(A, B, sa, sb, r)
    for call in range(3):
        got = _run(fl, A, B, sa, sb)
        assert_within_bound(got, r, bound, "tile pairs, call %d" % call)
        assert np.mean(got == oracle.bf16_bits_to_float(Cref)) > 0.98


def test_equal_scales_match_pertensor_bound():
    fl = lib()
    rng = np.random.default_rng(2)
    M, N, K = 256, 256, 512
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa = np.full((M // 32, K // 32), 0.25, np.float32)
    sb = np.full((N // 32, K // 32), 3.0, np.float32)
    got = _run(fl, A, B, sa, sb)
    check_pertensor(got, A, B, np.float32(0.25), np.float32(3.0), what="equal scales")


def test_one_hot_k_block():
    """Only K block 3 has nonzero scales: C is that block's product alone."""
    fl = lib()
    rng = np.random.default_rng(3)
    M, N, K = 128, 128, 256
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa = np.zeros((4, 8), np.float32)
    sb = np.ones((4, 8), np.float32)
    sa[:, 3] = 0.5
    # (N = 128 here, so sb has 4 column-tile rows)
    got = _run(fl, A, B, sa, sb)
    check_pertensor(got, A[:, 96:128], B[:, 96:128], np.float32(0.5), np.float32(1),
                    what="one-hot")


def test_k_zero_writes_zeros():
    import torch
    fl = lib()
    C = torch.full((64, 64), 1.0, dtype=torch.bfloat16, device="cuda")
    fl.fp8_gemm_blockscaled_32x32(0, 16, 0, 16, C.data_ptr(), 64, 64, 64, 0, 0, 1, 0, 1,
                                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.all(C == 0)


@pytest.mark.parametrize("name", ["qkv", "attn_out", "gate_up", "down"])
def test_transformer_linears_full_size_sampled(name):
    """M=4096 tokens through each 70B-class linear: 32x32 block quantisation
    of activations and weights on the GPU (checked against the oracle on
    sampled tiles), then the block-scaled GEMM checked on sampled outputs,
    on one whole 128-row tile row of C and on one whole 64-column tile
    column."""
    import torch
    fl = lib()
    X, W = workloads.transformer_linear(name, seed=0)
    qx, sx = fl.quantize_blockwise_32x32(to_dev(X))
    qw, sw = fl.quantize_blockwise_32x32(to_dev(W))
    C = fl.gemm_blockscaled_32x32(qx, qw, sx, sw)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    A, B = qx.cpu().numpy(), qw.cpu().numpy()
    sa, sb = sx.cpu().numpy(), sw.cpu().numpy()
    rng = np.random.default_rng(11)
    # quantiser parity on sampled 64x64 regions
    for (src, q, s) in ((X, A, sa), (W, B, sb)):
        r0 = int(rng.integers(0, src.shape[0] // 32 - 1)) * 32
        c0 = int(rng.integers(0, src.shape[1] // 32 - 1)) * 32
        rq, rs = oracle.quantize_blockwise_32x32(src[r0:r0 + 64, c0:c0 + 64])
        assert np.array_equal(q[r0:r0 + 64, c0:c0 + 64], rq)
        assert np.array_equal(s[r0 // 32:r0 // 32 + 2, c0 // 32:c0 // 32 + 2], rs)
    maxes = (oracle.max_abs_tile_scaled_32x32(A, sa), oracle.max_abs_tile_scaled_32x32(B, sb))
    rows = np.sort(rng.choice(A.shape[0], 64, replace=False))
    cols = np.sort(rng.choice(B.shape[0], 64, replace=False))
    Cn = bf16_to_f64(C[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()])
    check_block(Cn, A, B, sa, sb, rows=rows, cols=cols, what=name, maxes=maxes)
    # one whole 128-row tile row of C (every column tile, every K block) and
    # one whole 64-column tile column (every row tile), in bounded chunks
    M, N = C.shape
    r0 = int(rng.integers(0, M // 128)) * 128
    c0 = int(rng.integers(0, N // 64)) * 64
    Cg = C[r0:r0 + 128].float().cpu().numpy().astype(np.float64)
    step = max(512, (1 << 25) // A.shape[1])     # decoded B chunk <= 256 MB
    for j0 in range(0, N, step):
        cols = np.arange(j0, min(N, j0 + step))
        check_block(Cg[:, j0:j0 + cols.size], A, B, sa, sb, rows=np.arange(r0, r0 + 128),
                    cols=cols, what="%s rows %d.." % (name, r0), maxes=maxes)
    Cg = C[:, c0:c0 + 64].float().cpu().numpy().astype(np.float64)
    for i0 in range(0, M, 1024):
        rows = np.arange(i0, min(M, i0 + 1024))
        check_block(Cg[i0:i0 + rows.size], A, B, sa, sb, rows=rows,
                    cols=np.arange(c0, c0 + 64), what="%s cols %d.." % (name, c0), maxes=maxes)


def test_long_k_all_outputs():
    """K = 65530: 512 stages per tile (the 7-slot ring wraps 73 times), 2048
    scale blocks along K with a ragged last one; every output within the
    bound."""
    fl = lib()
    rng = np.random.default_rng(65530)
    M, N, K = 160, 200, 65530
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    nkb = -(-K // 32)
    sa = rng.uniform(1e-3, 2.0, (-(-M // 32), nkb)).astype(np.float32)
    sb = rng.uniform(1e-3, 2.0, (-(-N // 32), nkb)).astype(np.float32)
    got = _run(fl, A, B, sa, sb)
    frac = check_block(got, A, B, sa, sb, what="K %d" % K)
    assert frac > 0.9
