"""Run-to-run determinism of the GEMM kernels at full size: repeated calls on
the same inputs give the same BF16 bits, also when another kernel runs
beside them on a second stream (which changes the timing of every
hand-off inside the persistent kernels but none of their arithmetic)."""

import pytest

from _helpers import lib

pytestmark = pytest.mark.gpu


def _codes(torch, g, shape):
    """Uniform over the 254 finite E4M3 codes, generated on the device."""
    x = torch.randint(0, 254, shape, device="cuda", generator=g, dtype=torch.int16)
    return (x + (x >= 0x7F).to(torch.int16)).to(torch.uint8)


def _busy_side_stream(torch, fl, x, q, amax, scale):
    """Queue HBM-bound quantiser launches on a second stream."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(4):
            fl.quantize_pertensor(x, q, amax, scale)
    return side


def _repeat(torch, fl, run, n=3):
    """run() n times on the current stream, once more beside a busy second
    stream; every result must equal the first bit for bit."""
    first = run().view(torch.int16).clone()
    for _ in range(n - 1):
        assert torch.equal(run().view(torch.int16), first)
    x = torch.randn(8192, 8192, device="cuda")
    q = torch.empty(8192, 8192, dtype=torch.uint8, device="cuda")
    amax = torch.empty(1, device="cuda")
    scale = torch.empty(1, device="cuda")
    side = _busy_side_stream(torch, fl, x, q, amax, scale)
    out = run().view(torch.int16)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    assert torch.equal(out, first)


@pytest.mark.parametrize("variant", [0, 1, 2, 4])
def test_pertensor_8192(variant):
    import torch
    fl = lib()
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    A = _codes(torch, g, (8192, 8192))
    B = _codes(torch, g, (8192, 8192))
    sa = torch.tensor([0.003], device="cuda")
    sb = torch.tensor([0.002], device="cuda")
    C = torch.empty(8192, 8192, dtype=torch.bfloat16, device="cuda")
    fl.fp8la_set_gemm_variant(variant)
    try:
        _repeat(torch, fl, lambda: fl.gemm(A, B, sa, sb, C))
    finally:
        fl.fp8la_set_gemm_variant(0)


def test_blockscaled_attn_out():
    import torch
    fl = lib()
    g = torch.Generator(device="cuda")
    g.manual_seed(12)
    M, N, K = 4096, 8192, 8192
    A = _codes(torch, g, (M, K))
    B = _codes(torch, g, (N, K))
    sa = torch.rand(M // 32, K // 32, device="cuda", generator=g) + 0.5
    sb = torch.rand(N // 32, K // 32, device="cuda", generator=g) + 0.5
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    _repeat(torch, fl, lambda: fl.gemm_blockscaled_32x32(A, B, sa, sb, C))


def test_grouped_moe():
    import numpy as np
    import torch
    from precision_linear_algebra_gb300 import workloads
    fl = lib()
    counts, _ = workloads.moe_counts(seed=0)
    offs = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).cuda()
    E, N, K = len(counts), 14336, 4096
    g = torch.Generator(device="cuda")
    g.manual_seed(13)
    A = _codes(torch, g, (int(counts.sum()), K))
    B = _codes(torch, g, (E, N, K))
    sa = torch.rand(E, device="cuda", generator=g) * 0.01
    sb = torch.rand(E, device="cuda", generator=g) * 0.01
    C = torch.empty(A.shape[0], N, dtype=torch.bfloat16, device="cuda")
    _repeat(torch, fl, lambda: fl.grouped_gemm(offs, A, B, sa, sb, C))
