"""Pins for the oracle's delayed-scaling quantiser (CPU only).

Delayed scaling quantises with the scale of an amax carried over from an
earlier call and records the current tensor's amax for the next one.  Pins:
hand-worked codes, saturation when the tensor outgrows the carried-over
amax, the amax = 0 case against torch's own E4M3 cast, the reduction to
current scaling when the carried-over amax is the tensor's own, and the
scale as an IEEE fp32 division computed by torch.
"""

import numpy as np
import pytest
import torch

import oracle


def test_hand_example():
    x = np.array([1.0, -2.0, 0.5, 0.0], dtype=np.float32)
    q, amax, scale = oracle.quantize_pertensor_delayed(x, 4.0)
    # qscale = 448 / 4 = 112: 112 = 1.75*2^6 -> 0x6E, -224 = -1.75*2^7 -> 0xF6,
    # 56 = 1.75*2^5 -> 0x66, 0 -> 0x00; the recorded amax is the tensor's own.
    assert q.tolist() == [0x6E, 0xF6, 0x66, 0x00]
    assert amax == np.float32(2.0)
    assert scale == np.float32(4.0) / np.float32(448.0)


def test_saturates_beyond_carried_amax():
    x = np.array([2.0, -3.0, 0.5], dtype=np.float32)
    q, amax, scale = oracle.quantize_pertensor_delayed(x, 1.0)
    # qscale = 448: 896 and -1344 clamp to +-448, 224 -> 0x76
    assert q.tolist() == [0x7E, 0xFE, 0x76]
    assert amax == np.float32(3.0) and scale == np.float32(1.0 / 448.0)


def test_zero_carried_amax_is_unit_scale():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(4096) * 50).astype(np.float32)
    x = np.clip(x, -440, 440)
    q, amax, scale = oracle.quantize_pertensor_delayed(x, 0.0)
    assert scale == 1.0
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, want)
    assert amax == np.float32(np.abs(x).max())


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_own_amax_reduces_to_current_scaling(fmt):
    rng = np.random.default_rng(12)
    for trial in range(20):
        x = (rng.standard_normal((33, 65)) * 10.0 ** rng.uniform(-8, 8)).astype(np.float32)
        qc, amax_c, scale_c = oracle.quantize_pertensor(x, fmt)
        qd, amax_d, scale_d = oracle.quantize_pertensor_delayed(x, amax_c, fmt)
        assert np.array_equal(qc, qd) and amax_c == amax_d and scale_c == scale_d


def test_scale_is_fp32_division():
    for a in [3.0, 1e-3, 7.123, 1e20, 2.0 ** -100]:
        _, _, scale = oracle.quantize_pertensor_delayed(np.ones(3, np.float32), a)
        want = torch.tensor([float(np.float32(a))], dtype=torch.float32) / 448.0
        assert scale == np.float32(want.item())


def test_history_chain():
    """Two steps in a row: the second call's scale is the first call's amax."""
    rng = np.random.default_rng(13)
    x1 = rng.standard_normal(1000).astype(np.float32)
    x2 = (rng.standard_normal(1000) * 2).astype(np.float32)
    _, a1, _ = oracle.quantize_pertensor_delayed(x1, 0.0)
    q2, a2, s2 = oracle.quantize_pertensor_delayed(x2, a1)
    assert s2 == np.float32(a1) / np.float32(448.0)
    assert a2 == np.float32(np.abs(x2).max())
    # x2 has twice the spread, so some values exceed a1 and saturate
    assert np.any((q2 & 0x7F) == 0x7E)
