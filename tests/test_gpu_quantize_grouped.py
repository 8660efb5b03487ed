"""GPU parity: grouped per-tensor quantisation (each MoE expert's rows with
their own amax and scale, offsets on the device) against the oracle, bit for
bit: codes, amax and scale of every group.  Rows past the last group, and
columns past cols, come back untouched; offsets that break the rules are
reported and nothing is written."""

import numpy as np
import pytest

import oracle
from _helpers import lib, to_dev
from precision_linear_algebra_gb300 import workloads

pytestmark = pytest.mark.gpu

SENTINEL = 0xA5


def _run(fl, x_np, offs, cap_extra=0, ldx_pad=0, ldq_pad=0):
    import torch
    rows, cols = x_np.shape
    cap = rows + cap_extra
    xs = torch.zeros((cap, cols + ldx_pad), dtype=torch.float32, device="cuda")
    xs[:rows, :cols] = to_dev(x_np)
    qs = torch.full((cap, cols + ldq_pad), SENTINEL, dtype=torch.uint8, device="cuda")
    d_off = to_dev(np.asarray(offs, np.int32))
    E = len(offs) - 1
    scale = torch.full((E,), -1.0, dtype=torch.float32, device="cuda")
    q, amax, scale = fl.quantize_pertensor_grouped(xs[:, :cols], d_off, q=qs[:, :cols],
                                                   scale=scale)
    torch.cuda.synchronize()
    return qs.cpu().numpy(), amax.cpu().numpy(), scale.cpu().numpy(), fl.device_status()


def _check(got, x_np, offs, cols):
    qs, amax, scale, status = got
    assert status == 0
    rq, ramax, rscale = oracle.quantize_pertensor_grouped(x_np, offs)
    n = int(offs[-1])
    diff = np.argwhere(qs[:n, :cols] != rq)
    assert diff.size == 0, "codes differ at %d places, first (row, col) %s" % (
        len(diff), tuple(diff[0]))
    assert np.array_equal(amax.view(np.uint32), ramax.view(np.uint32))
    assert np.array_equal(scale.view(np.uint32), rscale.view(np.uint32))
    assert np.all(qs[n:] == SENTINEL), "rows past the last group written"
    assert np.all(qs[:, cols:] == SENTINEL), "columns past cols written"


@pytest.mark.parametrize("case", range(12))
def test_random_groups(case):
    fl = lib()
    rng = np.random.default_rng(500 + case)
    E = int(rng.integers(1, 10))
    counts = rng.integers(0, 300, E) * (rng.random(E) > 0.25)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    cols = int(rng.integers(1, 700))
    if case % 3 == 0:
        cols = cols // 4 * 4 + 4          # 16-byte rows
    x = (rng.standard_normal((int(offs[-1]), cols))
         * 10.0 ** rng.uniform(-3, 3, (int(offs[-1]), 1))).astype(np.float32)
    if x.size:
        x.reshape(-1)[rng.integers(0, x.size, 3)] = np.nan    # ignored by the amax
    pads = [(0, 0), (4, 8), (3, 5)][case % 3]
    _check(_run(fl, x, offs, cap_extra=int(rng.integers(0, 40)), ldx_pad=pads[0],
                ldq_pad=pads[1]), x, offs, cols)


def test_moe_activations_full_size():
    """The 16384 routed rows of the MoE layer (8 experts, K 4096)."""
    fl = lib()
    counts, offs, X, _ = workloads.moe_layer(seed=0)
    _check(_run(fl, X, offs), X, offs, X.shape[1])


def test_empty_groups_and_no_rows():
    fl = lib()
    x = np.zeros((0, 16), np.float32)
    qs, amax, scale, status = _run(fl, x, [0, 0, 0], cap_extra=8)
    assert status == 0
    assert np.array_equal(amax, [0.0, 0.0]) and np.array_equal(scale, [1.0, 1.0])
    assert np.all(qs == SENTINEL)


@pytest.mark.parametrize("offs", [[1, 8, 16], [0, 12, 8], [0, 8, 64]],
                         ids=["start_not_0", "decreasing", "past_capacity"])
def test_bad_offsets_write_nothing_and_are_reported(offs):
    fl = lib()
    rng = np.random.default_rng(9)
    x = rng.standard_normal((16, 40)).astype(np.float32)
    qs, amax, scale, status = _run(fl, x, offs, cap_extra=4)
    assert status == fl.FP8LA_ERR_DEVICE_ARG
    assert np.all(qs == SENTINEL), "codes written for bad offsets"
    assert np.all(scale == -1.0), "scales written for bad offsets"
