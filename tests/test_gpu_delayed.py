"""GPU parity: delayed-scaling quantiser (scale from a carried-over amax,
current amax recorded in one pass) against the oracle, bit for bit: codes,
recorded amax and scale."""

import numpy as np
import pytest

import oracle
from _helpers import lib, to_dev
from precision_linear_algebra_gb300 import workloads

pytestmark = pytest.mark.gpu


def _run(fl, x_np, amax_prev, fmt="e4m3", ldx_pad=0, ldq_pad=0):
    import torch
    rows, cols = x_np.shape
    xs = torch.empty((rows, cols + ldx_pad), dtype=torch.float32, device="cuda")
    xs[:, :cols] = to_dev(x_np)
    qs = torch.full((rows, cols + ldq_pad), 0xA5, dtype=torch.uint8, device="cuda")
    prev = torch.tensor([amax_prev], dtype=torch.float32, device="cuda")
    q, amax, scale = fl.quantize_pertensor_delayed(xs[:, :cols], prev, q=qs[:, :cols], fmt=fmt)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    if ldq_pad:
        assert torch.all(qs[:, cols:] == 0xA5), "write outside the row"
    return q.cpu().numpy(), amax.item(), scale.item()


def _check(got, x_np, amax_prev, fmt="e4m3"):
    q, amax, scale = got
    rq, ramax, rscale = oracle.quantize_pertensor_delayed(x_np, amax_prev, fmt)
    assert np.float32(amax).tobytes() == np.float32(ramax).tobytes()
    assert np.float32(scale).tobytes() == np.float32(rscale).tobytes()
    diff = np.flatnonzero(q.reshape(-1) != rq.reshape(-1))
    assert diff.size == 0, "codes differ at %d places, first %d: got %#x want %#x (x=%r)" % (
        diff.size, diff[0], q.reshape(-1)[diff[0]], rq.reshape(-1)[diff[0]],
        x_np.reshape(-1)[diff[0]])


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("shape,ldx_pad,ldq_pad", [
    ((1, 1), 0, 0), ((7, 13), 0, 0), ((33, 64), 0, 0), ((65, 100), 4, 16),
    ((3, 17), 3, 5), ((1000, 1001), 0, 0), ((512, 4096), 0, 0)])
def test_ragged_strided_and_carried_amax(shape, ldx_pad, ldq_pad, fmt):
    fl = lib()
    rng = np.random.default_rng(hash((shape, fmt)) & 0xFFFF)
    x = (rng.standard_normal(shape) * 3).astype(np.float32)
    own = float(np.abs(x).max())
    # own amax (current scaling), a smaller one (saturation), a larger one, zero
    for prev in (own, own / 4, own * 3.7, 0.0):
        _check(_run(fl, x, prev, fmt, ldx_pad, ldq_pad), x, prev, fmt)


def test_full_size_operands():
    """The 8192 x 8192 operands of the headline workload, carried-over amax
    from the other operand (so one saturates and one does not)."""
    fl = lib()
    A, B = workloads.square_outliers(8192, seed=0)
    aa, ab = float(np.abs(A).max()), float(np.abs(B).max())
    for x, prev in ((A, ab), (B, aa)):
        _check(_run(fl, x, prev), x, prev)


def test_history_chain_two_words():
    """Steps in a row through the C-ABI, alternating two amax words: each
    step's scale comes from the previous step's recorded amax."""
    import torch
    fl = lib()
    rng = np.random.default_rng(21)
    xs = [(rng.standard_normal((256, 384)) * (1 + i)).astype(np.float32) for i in range(4)]
    words = torch.zeros(2, dtype=torch.float32, device="cuda")
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    q = torch.empty((256, 384), dtype=torch.uint8, device="cuda")
    P = lambda t, i=0: t.data_ptr() + i * t.element_size()
    s = torch.cuda.current_stream().cuda_stream
    prev_host = 0.0
    for i, x_np in enumerate(xs):
        x = to_dev(x_np)
        cur, old = i & 1, (i & 1) ^ 1
        fl.fp8_quantize_pertensor_delayed(P(x), 256, 384, 384, P(q), 384, P(words, old),
                                          P(words, cur), P(scale), 0, s)
        torch.cuda.synchronize()
        _check((q.cpu().numpy(), words[cur].item(), scale.item()), x_np, prev_host)
        prev_host = words[cur].item()


def test_empty_and_aliasing():
    import torch
    fl = lib()
    words = torch.tensor([5.0, 7.0, 9.0], dtype=torch.float32, device="cuda")
    P = lambda t, i=0: t.data_ptr() + i * t.element_size()
    s = torch.cuda.current_stream().cuda_stream
    q = torch.empty(4, dtype=torch.uint8, device="cuda")
    x = torch.ones(4, dtype=torch.float32, device="cuda")
    fl.fp8_quantize_pertensor_delayed(P(x), 0, 4, 4, P(q), 4, P(words, 0), P(words, 1),
                                      P(words, 2), 0, s)
    torch.cuda.synchronize()
    assert words[1].item() == 0.0
    assert words[2].item() == np.float32(np.float32(5.0) / np.float32(448.0))
    st = fl.load().fp8_quantize_pertensor_delayed(P(x), 1, 4, 4, P(q), 4, P(words, 0),
                                                  P(words, 0), P(words, 2), 0, s)
    assert st == fl.FP8LA_ERR_INVALID_ARG


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_special_carried_amax_and_inputs(fmt):
    """Degenerate carried-over amax values (+Inf: qscale 0; NaN and fp32
    subnormals: qscale not finite, so qscale = scale = 1; the fp32 maximum)
    and inputs holding +-Inf, NaN, signed zeros and subnormals, whose
    recorded amax ignores the NaN and is Inf."""
    fl = lib()
    rng = np.random.default_rng(19)
    x = (rng.standard_normal((37, 90)) * 5).astype(np.float32)
    x[0, :6] = [np.inf, -np.inf, np.nan, 0.0, -0.0, 1e-42]
    x[36, 89] = np.nan
    clean = x.copy()
    clean[0, :3] = [1.0, -2.0, 3.0]
    for xx in (x, clean):
        for prev in (np.inf, np.nan, 1e-40, 3.4e38, 448.0):
            _check(_run(fl, xx, prev, fmt, 3, 8), xx, prev, fmt)
