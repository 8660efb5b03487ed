"""Failure detection without a GPU fault: a bounded in-kernel wait that
runs out must be reported through the device status word, and leave the
CUDA context usable.

The diagnostic entry point withholds the producer's first TMA arrival, so
the MMA warp's wait on that stage can never complete; with a 1 ms limit the
kernel records FP8LA_ERR_DEVICE_TIMEOUT, the other warps see the abort
flag, tensor memory is freed and the kernel returns."""

import numpy as np
import pytest

from _helpers import (assert_within_bound, bf16_to_f64, check_pertensor, lib, random_codes,
                      to_dev)

pytestmark = pytest.mark.gpu


def test_withheld_arrival_times_out_and_context_survives():
    import torch
    fl = lib()
    rng = np.random.default_rng(0)
    A = random_codes(rng, (128, 128))
    B = random_codes(rng, (256, 128))
    dA, dB = to_dev(A), to_dev(B)
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    C = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert fl.fp8_get_device_status(stream) == 0
    fl.fp8la_set_wait_timeout_ns(1_000_000)
    try:
        fl.fp8la_diag_gemm_withheld_arrival(dA.data_ptr(), 128, dB.data_ptr(), 128,
                                            C.data_ptr(), 256, one.data_ptr(),
                                            one.data_ptr(), stream)
        assert fl.fp8_get_device_status(stream) == fl.FP8LA_ERR_DEVICE_TIMEOUT
        # the status word was cleared by the read
        assert fl.fp8_get_device_status(stream) == 0
    finally:
        fl.fp8la_set_wait_timeout_ns(2_000_000_000)
    # the context is still usable: a normal GEMM runs and is correct
    C2 = fl.gemm(dA, dB, one, one)
    torch.cuda.synchronize()
    assert fl.fp8_get_device_status(stream) == 0
    check_pertensor(bf16_to_f64(C2), A, B, np.float32(1), np.float32(1), what="after timeout")


def _timeout_then(fl, launch):
    """Run `launch` with a 1 ms wait limit; it must report a timeout."""
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    assert fl.fp8_get_device_status(stream) == 0
    fl.fp8la_set_wait_timeout_ns(1_000_000)
    try:
        launch(stream)
        assert fl.fp8_get_device_status(stream) == fl.FP8LA_ERR_DEVICE_TIMEOUT
        assert fl.fp8_get_device_status(stream) == 0
    finally:
        fl.fp8la_set_wait_timeout_ns(2_000_000_000)


def test_cta_pair_withheld_arrival_times_out_and_context_survives():
    """The second CTA of the pair leaves out its first loads: the leader's
    MMA wait runs out, then the second CTA's own waits; both CTAs meet at
    the final cluster barrier, free their tensor memory and return."""
    import torch
    fl = lib()
    rng = np.random.default_rng(1)
    M, N, K = 256, 512, 384
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    dA, dB = to_dev(A), to_dev(B)
    sa = torch.full((1,), 0.5, dtype=torch.float32, device="cuda")
    sb = torch.full((1,), 0.25, dtype=torch.float32, device="cuda")
    C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    _timeout_then(fl, lambda s: fl.fp8la_diag_withheld_arrival(
        fl.FP8LA_DIAG_KERNEL_PAIR, dA.data_ptr(), K, dB.data_ptr(), K, C.data_ptr(), N,
        M, N, K, sa.data_ptr(), 0, sb.data_ptr(), 0, s))
    fl.fp8la_set_gemm_variant(2)
    try:
        C2 = fl.gemm(dA, dB, sa, sb)
    finally:
        fl.fp8la_set_gemm_variant(0)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    check_pertensor(bf16_to_f64(C2), A, B, np.float32(0.5), np.float32(0.25),
                    what="CTA pair after timeout")


def test_block_scaled_withheld_arrival_times_out_and_context_survives():
    """The block-scaled producer leaves out its first stage: the MMA and
    promotion warps' waits run out, the kernel drains and returns."""
    import torch
    import oracle
    fl = lib()
    rng = np.random.default_rng(2)
    M, N, K = 256, 192, 320
    A, B = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa = rng.uniform(0.01, 2, (M // 32, K // 32)).astype(np.float32)
    sb = rng.uniform(0.01, 2, (N // 32, K // 32)).astype(np.float32)
    dA, dB = to_dev(A), to_dev(B)
    ld = (K // 32 + 3) // 4 * 4
    dsa = torch.zeros((M // 32, ld), dtype=torch.float32, device="cuda")
    dsb = torch.zeros((N // 32, ld), dtype=torch.float32, device="cuda")
    dsa[:, :K // 32] = to_dev(sa)
    dsb[:, :K // 32] = to_dev(sb)
    C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    _timeout_then(fl, lambda s: fl.fp8la_diag_withheld_arrival(
        fl.FP8LA_DIAG_KERNEL_BLOCK32, dA.data_ptr(), K, dB.data_ptr(), K, C.data_ptr(), N,
        M, N, K, dsa.data_ptr(), ld, dsb.data_ptr(), ld, s))
    C2 = fl.gemm_blockscaled_32x32(dA, dB, dsa[:, :K // 32], dsb[:, :K // 32])
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    r, _ = oracle.gemm_blockscaled_32x32(A, B, sa, sb)
    assert_within_bound(bf16_to_f64(C2), r, oracle.tolerance_blockscaled_32x32(A, B, sa, sb, r),
                        "block-scaled after timeout")
