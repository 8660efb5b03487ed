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


def test_special_value_groups():
    """Groups holding the degenerate cases of the scale rule: zeros, signed
    zeros, +Inf (amax Inf: qscale 0, scale Inf), NaN beside finite values,
    NaN only (amax 0), fp32 subnormals only (448/amax overflows: qscale =
    scale = 1), values near the fp32 maximum, and an ordinary group."""
    fl = lib()
    rng = np.random.default_rng(31)
    cols = 72
    parts = [np.zeros((5, cols), np.float32),
             np.full((3, cols), -0.0, np.float32),
             rng.standard_normal((9, cols)).astype(np.float32),
             rng.standard_normal((4, cols)).astype(np.float32),
             np.full((2, cols), np.nan, np.float32),
             (rng.standard_normal((6, cols)) * 1e-40).astype(np.float32),
             (rng.uniform(-3.0, 3.0, (7, cols)) * 1e38).astype(np.float32),
             (rng.standard_normal((11, cols)) * 0.02).astype(np.float32)]
    parts[2][4, 5] = np.inf
    parts[3][1, :3] = np.nan
    parts[6][0, 0] = np.float32(3.4e38)
    x = np.concatenate(parts)
    offs = np.concatenate([[0], np.cumsum([p.shape[0] for p in parts])]).astype(np.int32)
    got = _run(fl, x, offs, cap_extra=6, ldx_pad=4, ldq_pad=8)
    _check(got, x, offs, cols)
    _, amax, scale, _ = got
    assert amax[0] == 0 and scale[0] == 1 and scale[2] == np.inf and amax[4] == 0
    assert scale[5] == 1 and np.isfinite(scale[6])


def test_maximum_group_count():
    """1024 groups, the largest the header allows, most of them empty."""
    fl = lib()
    rng = np.random.default_rng(4096)
    E, cols = 1024, 40
    counts = np.zeros(E, np.int64)
    idx = rng.choice(E, 80, replace=False)
    counts[idx] = rng.integers(1, 9, 80)
    counts[777] = 300
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = (rng.standard_normal((int(offs[-1]), cols))
         * 10.0 ** rng.uniform(-3, 3, (int(offs[-1]), 1))).astype(np.float32)
    _check(_run(fl, x, offs, cap_extra=9, ldx_pad=4, ldq_pad=8), x, offs, cols)
