"""GPU parity: grouped (MoE) E4M3 GEMM against the oracle, per group within
the per-tensor bound with that group's scales; rows outside every group are
left untouched."""

import numpy as np
import pytest

import oracle
from _helpers import bf16_to_f64, check_pertensor, lib, random_codes, to_dev
from precision_linear_algebra_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[1, 2], ids=["single_cta", "cta_pair"])
def variant(request):
    fl = lib()
    fl.fp8la_set_gemm_variant(request.param)
    yield request.param
    fl.fp8la_set_gemm_variant(0)


def _grouped(fl, A, offs, B, sa, sb, cap_extra=0):
    import torch
    cap = A.shape[0] + cap_extra
    K = A.shape[1]
    E, N, _ = B.shape
    kp = max(16, (K + 15) // 16 * 16)
    dA = torch.zeros((cap, kp), dtype=torch.uint8, device="cuda")
    dA[:A.shape[0], :K] = to_dev(A)
    dB = torch.zeros((E, N, kp), dtype=torch.uint8, device="cuda")
    dB[:, :, :K] = to_dev(B)
    dC = torch.full((cap, N), 3.0, dtype=torch.bfloat16, device="cuda")
    d_off = to_dev(np.asarray(offs, np.int32))
    d_sa = to_dev(np.asarray(sa, np.float32))
    d_sb = to_dev(np.asarray(sb, np.float32))
    fl.fp8_grouped_gemm(E, d_off.data_ptr(), cap, dA.data_ptr(), kp, dB.data_ptr(), kp,
                        N * kp, dC.data_ptr(), N, N, K, d_sa.data_ptr(), d_sb.data_ptr(),
                        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    return bf16_to_f64(dC)


@pytest.mark.parametrize("counts,N,K", [
    ([7, 0, 300, 0, 129], 512, 256),
    ([128, 128], 256, 128),
    ([0, 0, 1], 96, 48),
    ([1000], 600, 200),
    ([5, 17, 250, 3, 0, 0, 140, 77], 272, 160),
])
def test_grouped_random_codes(counts, N, K, variant):
    fl = lib()
    rng = np.random.default_rng(sum(counts) + N + K)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    E = len(counts)
    A = random_codes(rng, (int(offs[-1]), K))
    B = random_codes(rng, (E, N, K))
    sa = rng.uniform(0.01, 2, E).astype(np.float32)
    sb = rng.uniform(0.01, 2, E).astype(np.float32)
    got = _grouped(fl, A, offs, B, sa, sb, cap_extra=37)
    for e in range(E):
        lo, hi = offs[e], offs[e + 1]
        if hi > lo:
            check_pertensor(got[lo:hi], A[lo:hi], B[e], sa[e], sb[e], what="group %d" % e)
    assert np.all(got[offs[-1]:] == 3.0), "rows past the last group were written"


def test_grouped_equals_per_group_gemm_calls(variant):
    """One grouped launch equals E separate fp8_gemm calls, bit for bit."""
    import torch
    fl = lib()
    rng = np.random.default_rng(12)
    counts = [200, 0, 64, 333]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    N, K = 512, 384
    A = random_codes(rng, (int(offs[-1]), K))
    B = random_codes(rng, (4, N, K))
    sa = rng.uniform(0.1, 1, 4).astype(np.float32)
    sb = rng.uniform(0.1, 1, 4).astype(np.float32)
    got = _grouped(fl, A, offs, B, sa, sb)
    for e in range(4):
        lo, hi = offs[e], offs[e + 1]
        if hi == lo:
            continue
        C = fl.gemm(to_dev(A[lo:hi]), to_dev(B[e]), to_dev(sa[e:e + 1]), to_dev(sb[e:e + 1]))
        torch.cuda.synchronize()
        assert np.array_equal(bf16_to_f64(C), got[lo:hi])


def test_moe_layer_full_size_sampled(variant):
    """8 experts, K 4096, N 14336, 16384 routed rows with Dirichlet counts;
    per-expert per-tensor quantisation on the GPU, one grouped launch; the
    oracle checks sampled rows of every group against sampled columns, and
    every row of each group's first and last 256-row blocks (the last one
    partial, computed transposed by the CTA-pair kernel) against a
    contiguous 512-column block."""
    import torch
    fl = lib()
    counts, offs, X, W = workloads.moe_layer(seed=0)
    E, N, K = W.shape
    dX = to_dev(X)
    dW = to_dev(W)
    qx = torch.empty(X.shape, dtype=torch.uint8, device="cuda")
    qw = torch.empty(W.shape, dtype=torch.uint8, device="cuda")
    amax = torch.empty(2 * E, dtype=torch.float32, device="cuda")
    sx = torch.empty(E, dtype=torch.float32, device="cuda")
    sw = torch.empty(E, dtype=torch.float32, device="cuda")
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        fl.quantize_pertensor(dX[lo:hi], q=qx[lo:hi], amax=amax[e:e + 1], scale=sx[e:e + 1])
        fl.quantize_pertensor(dW[e], q=qw[e], amax=amax[E + e:E + e + 1], scale=sw[e:e + 1])
    C = fl.grouped_gemm(to_dev(offs), qx, qw, sx, sw)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    qx_n, qw_n, sx_n, sw_n = qx.cpu().numpy(), qw.cpu().numpy(), sx.cpu().numpy(), sw.cpu().numpy()
    Cn = bf16_to_f64(C)
    rng = np.random.default_rng(1)
    cols = np.sort(rng.choice(N, 96, replace=False))
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            continue
        rq, _, rs = oracle.quantize_pertensor(X[lo:hi])
        assert np.array_equal(qx_n[lo:hi], rq) and sx_n[e] == rs
        # weights: the oracle's amax and scales on the whole expert, its
        # cast on the sampled rows only (the cast is elementwise)
        qs, ws = oracle.scales_from_amax(oracle.amax_fp32(W[e]))
        assert sw_n[e] == ws
        assert np.array_equal(qw_n[e][cols], oracle.encode((W[e][cols] * qs).astype(np.float32)))
        rows = np.sort(rng.choice(hi - lo, min(48, hi - lo), replace=False))
        check_pertensor(Cn[lo + rows][:, cols], qx_n[lo:hi], qw_n[e], sx_n[e], sw_n[e],
                        rows=rows, cols=cols, what="expert %d" % e)
        n_rows = hi - lo
        last0 = (n_rows - 1) // 256 * 256
        rblk = np.unique(np.concatenate([np.arange(min(256, n_rows)),
                                         np.arange(last0, n_rows)]))
        c0 = int(rng.integers(0, N // 256 - 1)) * 256
        cblk = np.arange(c0, c0 + 512)
        assert np.array_equal(qw_n[e][cblk], oracle.encode((W[e][cblk] * qs).astype(np.float32)))
        check_pertensor(Cn[lo + rblk][:, cblk], qx_n[lo:hi], qw_n[e], sx_n[e], sw_n[e],
                        rows=rblk, cols=cblk,
                        what="expert %d, first and last row blocks" % e)


def _launch_raw(fl, E, d_off, cap, dA, kp, dB, N, dC, ldc, K, d_sa, d_sb):
    import torch
    fl.fp8_grouped_gemm(E, d_off.data_ptr(), cap, dA.data_ptr(), kp, dB.data_ptr(), kp,
                        N * kp, dC.data_ptr(), ldc, N, K, d_sa.data_ptr(), d_sb.data_ptr(),
                        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("offsets", [
    [0, 100, 200, 256 + 40],          # last offset past m_capacity (256)
    [0, 120, 60, 200],                # a decreasing pair
    [8, 100, 150, 200],               # does not start at 0
    [0, 300, 280, 256],               # past capacity inside, back at the end
], ids=["past_capacity", "decreasing", "nonzero_start", "overshoot_inside"])
@pytest.mark.parametrize("K", [128, 0], ids=["K128", "K0"])
def test_bad_offsets_write_nothing_and_are_reported(offsets, K, variant):
    """m_offsets that break the contract are caught on the device: nothing is
    written (C and guard rows past m_capacity, in the same allocation, keep
    their sentinel), the status word says FP8LA_ERR_DEVICE_ARG, and a valid
    call right after is correct."""
    import torch
    fl = lib()
    rng = np.random.default_rng(77)
    E, N, cap, guard = 3, 256, 256, 64
    kp = 128
    A = random_codes(rng, (cap + guard, kp))
    B = random_codes(rng, (E, N, kp))
    dA, dB = to_dev(A), to_dev(B)
    dC = torch.full((cap + guard, N), 7.0, dtype=torch.bfloat16, device="cuda")
    d_sa = to_dev(np.full(E, 0.5, np.float32))
    d_sb = to_dev(np.full(E, 0.25, np.float32))
    stream = torch.cuda.current_stream().cuda_stream
    assert fl.fp8_get_device_status(stream) == 0
    _launch_raw(fl, E, to_dev(np.asarray(offsets, np.int32)), cap, dA, kp, dB, N, dC, N,
                K, d_sa, d_sb)
    assert fl.fp8_get_device_status(stream) == fl.FP8LA_ERR_DEVICE_ARG
    assert fl.fp8_get_device_status(stream) == 0          # cleared by the read
    assert torch.all(dC == 7.0), "a call with bad offsets wrote to C"
    # the same buffers with valid offsets
    good = np.array([0, 100, 100, 230], np.int32)
    _launch_raw(fl, E, to_dev(good), cap, dA, kp, dB, N, dC, N, kp, d_sa, d_sb)
    assert fl.fp8_get_device_status(stream) == 0
    got = bf16_to_f64(dC)
    for e in range(E):
        lo, hi = good[e], good[e + 1]
        if hi > lo:
            check_pertensor(got[lo:hi], A[lo:hi], B[e], np.float32(0.5), np.float32(0.25),
                            what="group %d after bad offsets" % e)
    assert np.all(got[good[-1]:] == 7.0)


def test_rows_past_the_last_group_are_ignored(variant):
    """Rows of A past m_offsets[E] hold NaN codes (0x7F) and trailing groups
    are empty: the valid rows match the oracle, no NaN leaks in, and C rows
    past m_offsets[E] keep their sentinel."""
    import torch
    fl = lib()
    rng = np.random.default_rng(78)
    counts = [70, 0, 260, 3] + [0] * 12
    E = len(counts)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    N, K, cap = 320, 192, 700
    A = np.full((cap, K), 0x7F, np.uint8)
    A[:offs[-1]] = random_codes(rng, (int(offs[-1]), K))
    B = random_codes(rng, (E, N, K))
    dA, dB = to_dev(A), to_dev(B)
    dC = torch.full((cap, N), -2.0, dtype=torch.bfloat16, device="cuda")
    sa = rng.uniform(0.1, 2, E).astype(np.float32)
    sb = rng.uniform(0.1, 2, E).astype(np.float32)
    _launch_raw(fl, E, to_dev(offs), cap, dA, K, dB, N, dC, N, K, to_dev(sa), to_dev(sb))
    assert fl.device_status() == 0
    got = bf16_to_f64(dC)
    for e in range(E):
        lo, hi = offs[e], offs[e + 1]
        if hi > lo:
            check_pertensor(got[lo:hi], A[lo:hi], B[e], sa[e], sb[e], what="group %d" % e)
    assert np.all(got[offs[-1]:] == -2.0)


@pytest.mark.parametrize("N,K", [(300, 192), (512, 128)])
def test_tail_tiles_of_every_size(N, K, variant):
    """Groups whose last row tile holds 1..255 rows (the CTA-pair kernel
    computes tails of at most 128 rows transposed), N not a multiple of the
    tile width; every group against the oracle, rows past the last group
    untouched."""
    fl = lib()
    rng = np.random.default_rng(N + K)
    counts = [1, 16, 31, 32, 33, 64, 96, 100, 127, 128, 129, 255, 256, 257, 300, 0, 513]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    E = len(counts)
    A = random_codes(rng, (int(offs[-1]), K))
    B = random_codes(rng, (E, N, K))
    sa = rng.uniform(0.01, 2, E).astype(np.float32)
    sb = rng.uniform(0.01, 2, E).astype(np.float32)
    got = _grouped(fl, A, offs, B, sa, sb, cap_extra=45)
    for e in range(E):
        lo, hi = offs[e], offs[e + 1]
        if hi > lo:
            check_pertensor(got[lo:hi], A[lo:hi], B[e], sa[e], sb[e], what="group %d" % e)
    assert np.all(got[offs[-1]:] == 3.0), "rows past the last group were written"


def test_maximum_group_count(variant):
    """num_groups = 1024, the largest the header allows: most groups empty,
    some of one to a few rows, a few spanning several row tiles, the last
    groups empty; each expert's own scales; every nonempty group against the
    oracle and rows past the last group untouched."""
    fl = lib()
    rng = np.random.default_rng(1024)
    E, N, K = 1024, 96, 64
    counts = np.zeros(E, np.int64)
    small = rng.choice(E - 8, 60, replace=False)
    counts[small] = rng.integers(1, 5, 60)
    counts[[3, 500, 1000]] = [130, 257, 31]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    A = random_codes(rng, (int(offs[-1]), K))
    B = random_codes(rng, (E, N, K))
    sa = rng.uniform(0.01, 2, E).astype(np.float32)
    sb = rng.uniform(0.01, 2, E).astype(np.float32)
    got = _grouped(fl, A, offs, B, sa, sb, cap_extra=21)
    for e in np.flatnonzero(counts):
        lo, hi = offs[e], offs[e + 1]
        check_pertensor(got[lo:hi], A[lo:hi], B[e], sa[e], sb[e], what="group %d" % e)
    assert np.all(got[offs[-1]:] == 3.0), "rows past the last group were written"


def test_k_zero_writes_zeros_in_groups_only():
    """K = 0: every row inside a group becomes zero, with the offsets read on
    the device; rows past the last group keep their sentinel."""
    import torch
    fl = lib()
    counts = [5, 0, 130, 1]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    E, N, cap = len(counts), 72, 160
    dC = torch.full((cap, N), 3.0, dtype=torch.bfloat16, device="cuda")
    dA = torch.zeros((cap, 16), dtype=torch.uint8, device="cuda")
    dB = torch.zeros((E, N, 16), dtype=torch.uint8, device="cuda")
    ones = torch.ones(E, dtype=torch.float32, device="cuda")
    d_off = to_dev(offs)
    fl.fp8_grouped_gemm(E, d_off.data_ptr(), cap, dA.data_ptr(), 16, dB.data_ptr(), 16,
                        N * 16, dC.data_ptr(), N, N, 0, ones.data_ptr(), ones.data_ptr(),
                        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    got = bf16_to_f64(dC)
    assert np.all(got[:offs[-1]] == 0)
    assert np.all(got[offs[-1]:] == 3.0)


def test_long_k(variant):
    """K = 65536 over three groups (one empty): hundreds of laps of the
    stage ring per tile, every output within the bound."""
    fl = lib()
    rng = np.random.default_rng(65536)
    counts = [150, 0, 70]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    E, N, K = len(counts), 136, 65536
    A = random_codes(rng, (int(offs[-1]), K))
    B = random_codes(rng, (E, N, K))
    sa = rng.uniform(0.01, 2, E).astype(np.float32)
    sb = rng.uniform(0.01, 2, E).astype(np.float32)
    got = _grouped(fl, A, offs, B, sa, sb, cap_extra=10)
    for e in (0, 2):
        lo, hi = offs[e], offs[e + 1]
        check_pertensor(got[lo:hi], A[lo:hi], B[e], sa[e], sb[e], what="group %d" % e)
    assert np.all(got[offs[-1]:] == 3.0)
