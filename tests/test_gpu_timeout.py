"""Failure detection without a GPU fault: a bounded in-kernel wait that
runs out must be reported through the device status word, and leave the
CUDA context usable.

The diagnostic entry point withholds the producer's first TMA arrival, so
the MMA warp's wait on that stage can never complete; with a 1 ms limit the
kernel records FP8LA_ERR_DEVICE_TIMEOUT, the other warps see the abort
flag, tensor memory is freed and the kernel returns."""

import numpy as np
import pytest

from _helpers import bf16_to_f64, check_pertensor, lib, random_codes, to_dev

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
