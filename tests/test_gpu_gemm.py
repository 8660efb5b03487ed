"""GPU parity: per-tensor-scaled E4M3 GEMM against the oracle, within the bound

    |C_gpu - C_ref| <= 2^-8 |C_ref| + 2^-22 K sa sb max|a| max|b|

elementwise, C_ref being the oracle's exact product before its BF16 rounding
(see the oracle's bound_pertensor)."""

import numpy as np
import pytest

import oracle
from _helpers import bf16_to_f64, check_pertensor, lib, random_codes, to_dev
from precision_linear_algebra_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[1, 2, 3, 4], ids=["single_cta", "cta_pair", "single_cta_128", "cta_quad"])
def variant(request):
    """Run a test once per GEMM kernel (single-CTA 128 x 256 tiles, CTA
    pair, single-CTA 128 x 128 tiles, two CTA pairs per cluster sharing A
    by multicast)."""
    fl = lib()
    fl.fp8la_set_gemm_variant(request.param)
    yield request.param
    fl.fp8la_set_gemm_variant(0)


def _gemm(fl, A, B, sa, sb, ldc_pad=0):
    import torch
    M, K = A.shape
    N = B.shape[0]
    # TMA wants 16-byte row strides: pad K up to a multiple of 16
    kp = max(16, (K + 15) // 16 * 16)
    dA = torch.zeros((M, kp), dtype=torch.uint8, device="cuda")
    dB = torch.zeros((N, kp), dtype=torch.uint8, device="cuda")
    dA[:, :K] = to_dev(A)
    dB[:, :K] = to_dev(B)
    dA, dB = dA[:, :K], dB[:, :K]
    dsa = torch.tensor([sa], dtype=torch.float32, device="cuda")
    dsb = torch.tensor([sb], dtype=torch.float32, device="cuda")
    Cs = torch.full((M, N + ldc_pad), -7.0, dtype=torch.bfloat16, device="cuda")
    C = Cs[:, :N]
    fl.gemm(dA, dB, dsa, dsb, C=C)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    if ldc_pad:
        assert torch.all(Cs[:, N:] == -7.0), "write past N"
    return bf16_to_f64(C.contiguous())


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 128),    # one tile, one K block
    (128, 256, 32),     # K shorter than one K block
    (128, 256, 48),
    (128, 256, 16),
    (256, 512, 512),    # several tiles and K blocks
    (128, 256, 1024),   # K blocks beyond the pipeline depth
    (300, 270, 200),    # ragged M, N, K
    (1, 1, 16),
    (17, 8, 16),
    (129, 257, 144),
    (640, 1280, 384),
])
def test_random_codes(M, N, K, variant):
    fl = lib()
    rng = np.random.default_rng(M * 7 + N * 13 + K)
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa, sb = np.float32(0.37), np.float32(1.9)
    got = _gemm(fl, A, B, sa, sb)
    frac = check_pertensor(got, A, B, sa, sb, what="%dx%dx%d" % (M, N, K))
    assert frac > 0.99


def test_many_tiles_per_cta_all_outputs(variant):
    """About two 256 x 256 tiles per CTA pair (4096 x 2560) with ragged N and
    every output checked, so that tile changes, both TMEM accumulators and
    the edge-block stores are all exercised."""
    fl = lib()
    rng = np.random.default_rng(99)
    M, N, K = 4096, 2520, 256
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    got = _gemm(fl, A, B, np.float32(0.03125), np.float32(2.0), ldc_pad=8)
    frac = check_pertensor(got, A, B, np.float32(0.03125), np.float32(2.0), what="many tiles")
    assert frac > 0.98


def test_identity_operand_selects_columns(variant):
    """A = I (code 0x38 = 1): C = dec(B)^T exactly (every E4M3 value is a bf16)."""
    fl = lib()
    rng = np.random.default_rng(3)
    K = 128
    A = np.where(np.eye(K, dtype=bool), 0x38, 0).astype(np.uint8)
    B = random_codes(rng, (256, K))
    got = _gemm(fl, A, B, np.float32(1), np.float32(1))
    assert np.array_equal(got, oracle.decode(B).T)


def test_one_hot_rows_and_ldc_padding(variant):
    fl = lib()
    rng = np.random.default_rng(4)
    M, N, K = 200, 300, 256
    A = np.zeros((M, K), np.uint8)
    A[np.arange(M), rng.integers(0, K, M)] = 0x40            # 2.0 at one k per row
    B = random_codes(rng, (N, K))
    got = _gemm(fl, A, B, np.float32(0.5), np.float32(1), ldc_pad=12)
    check_pertensor(got, A, B, np.float32(0.5), np.float32(1), what="one-hot")


def test_k_zero_writes_zeros():
    fl = lib()
    A = np.zeros((5, 0), np.uint8)
    B = np.zeros((9, 0), np.uint8)
    got = _gemm(fl, A, B, np.float32(1), np.float32(1))
    assert got.shape == (5, 9) and np.all(got == 0)


def test_saturated_operands(variant):
    fl = lib()
    M, N, K = 128, 256, 512
    A = np.full((M, K), 0x7E, np.uint8)
    B = np.full((N, K), 0xFE, np.uint8)
    got = _gemm(fl, A, B, np.float32(1), np.float32(1))
    assert np.all(got == -448.0 * 448.0 * K)


@pytest.mark.parametrize("n", [256, 1024])
def test_square_configs_end_to_end(n, variant):
    """Quantise N(0,1) operands on the GPU, then GEMM; check both steps."""
    import torch
    fl = lib()
    A, B = workloads.square(n, seed=0)
    qa, _, sa = fl.quantize_pertensor(to_dev(A))
    qb, _, sb = fl.quantize_pertensor(to_dev(B))
    C = fl.gemm(qa, qb, sa, sb)
    torch.cuda.synchronize()
    rqa, _, rsa = oracle.quantize_pertensor(A)
    rqb, _, rsb = oracle.quantize_pertensor(B)
    assert np.array_equal(qa.cpu().numpy(), rqa) and np.array_equal(qb.cpu().numpy(), rqb)
    assert sa.item() == rsa and sb.item() == rsb
    frac = check_pertensor(bf16_to_f64(C), rqa, rqb, rsa, rsb, what="square %d" % n)
    assert frac > 0.99


def test_8192_outliers_sampled(variant):
    """Full-size 8192^3 with outliers, in the launch configuration the
    benchmark times; the oracle checks 96 sampled rows x all columns plus
    all rows x 64 sampled columns."""
    import torch
    fl = lib()
    A, B = workloads.square_outliers(8192, seed=0)
    qa, _, sa = fl.quantize_pertensor(to_dev(A))
    qb, _, sb = fl.quantize_pertensor(to_dev(B))
    C = fl.gemm(qa, qb, sa, sb)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    qa_n, qb_n = qa.cpu().numpy(), qb.cpu().numpy()
    rqa, _, rsa = oracle.quantize_pertensor(A)
    rqb, _, rsb = oracle.quantize_pertensor(B)
    assert np.array_equal(qa_n, rqa) and np.array_equal(qb_n, rqb)
    Cn = bf16_to_f64(C)
    rng = np.random.default_rng(8)
    rows = np.sort(rng.choice(8192, 96, replace=False))
    cols = np.sort(rng.choice(8192, 64, replace=False))
    check_pertensor(Cn[rows], rqa, rqb, rsa, rsb, rows=rows, what="rows")
    check_pertensor(Cn[:, cols], rqa, rqb, rsa, rsb, cols=cols, what="cols")


@pytest.mark.parametrize("M,N,K,positive", [
    (300, 280, 131071, False),   # the longest K whose oracle sum is exact; ragged
    (256, 256, 65536, True),     # all-positive codes: no cancellation, the
                                 # FP32 accumulation error is largest relative
                                 # to the sum
])
def test_long_k_all_outputs(M, N, K, positive, variant):
    """Long reductions: about a thousand 128-wide K stages per tile, so the
    stage ring wraps hundreds of times; every output within the bound."""
    fl = lib()
    rng = np.random.default_rng(K + M)
    if positive:
        codes = np.arange(0x08, 0x7F, dtype=np.uint8)       # positive normals
        A, B = rng.choice(codes, (M, K)), rng.choice(codes, (N, K))
    else:
        A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa, sb = np.float32(0.0123), np.float32(0.731)
    got = _gemm(fl, A, B, sa, sb)
    frac = check_pertensor(got, A, B, sa, sb, what="K %d" % K)
    assert frac > 0.9


@pytest.mark.parametrize("M,N,K", [(1, 300, 682), (340, 1, 682), (1, 1, 37), (1, 1, 4096)])
def test_single_row_operands_unpadded(M, N, K):
    """A or B with one row, K not a multiple of 16, passed as a contiguous
    (unpadded) tensor through the torch-level call: a single row's stride
    never addresses memory, so the binding passes a valid TMA stride for it.
    A multi-row operand keeps a row stride padded to 16 bytes.  Every output
    matches the oracle within the bound."""
    import torch
    fl = lib()
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa, sb = np.float32(0.37), np.float32(1.9)

    def dev(x):
        if x.shape[0] == 1:
            return to_dev(x)                      # [1][K], stride K
        kp = (K + 15) // 16 * 16
        d = torch.zeros((x.shape[0], kp), dtype=torch.uint8, device="cuda")
        d[:, :K] = to_dev(x)
        return d[:, :K]

    C = fl.gemm(dev(A), dev(B), torch.tensor([sa], device="cuda"),
                torch.tensor([sb], device="cuda"))
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    check_pertensor(bf16_to_f64(C), A, B, sa, sb, what="%dx%dx%d" % (M, N, K))
