"""Pins for the oracle's per-tensor and 32x32 block quantisers (CPU only).

Pins: hand-worked examples, the invariant that the largest-magnitude element
always lands on +-448, a dequantisation error bound that follows from E4M3's
3 mantissa bits, and the special cases (all zeros, infinity, NaN, empty).
"""

import numpy as np
import torch

import oracle


def test_hand_example():
    x = np.array([[1.0, -2.0], [0.5, 0.0]], dtype=np.float32)
    q, amax, scale = oracle.quantize_pertensor(x)
    # amax = 2, qscale = 448/2 = 224, scale = 2/448 = 1/224 (fp32-rounded)
    assert amax == np.float32(2.0)
    assert scale == np.float32(2.0) / np.float32(448.0)
    # 224 = 1.75 * 2^7 -> 0x76 ; -448 -> 0xFE ; 112 = 1.75 * 2^6 -> 0x6E ; 0 -> 0x00
    assert q.tolist() == [[0x76, 0xFE], [0x6E, 0x00]]


def test_scale_is_fp32_division():
    for a in [3.0, 1e-3, 7.123, 1e20, 2.0 ** -100]:
        x = np.array([a, -a / 3], dtype=np.float32)
        _, amax, scale = oracle.quantize_pertensor(x)
        want = torch.tensor([float(np.float32(a))], dtype=torch.float32) / 448.0
        assert scale == np.float32(want.item())


def test_amax_element_lands_on_448():
    rng = np.random.default_rng(3)
    for trial in range(200):
        x = (rng.standard_normal(257) * 10.0 ** rng.uniform(-30, 30)).astype(np.float32)
        q, amax, _ = oracle.quantize_pertensor(x)
        i = int(np.argmax(np.abs(x)))
        assert q[i] & 0x7F == 0x7E


def test_dequantised_error_bound():
    """|dec(q)*scale - x| <= 2^-4 |x| (normals) or 2^-10 * scale (subnormals)."""
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(100_000) * 3).astype(np.float32)
    q, amax, scale = oracle.quantize_pertensor(x)
    y = oracle.decode(q) * float(scale)
    # in code units the normal step is 2^-3 of the binade, half of it 2^-4
    err = np.abs(y - x.astype(np.float64))
    bound = 2.0 ** -4 * np.abs(x) * (1 + 1e-6) + 2.0 ** -10 * float(scale)
    assert np.all(err <= bound)


def test_special_cases():
    z = np.zeros((3, 5), dtype=np.float32)
    q, amax, scale = oracle.quantize_pertensor(z)
    assert amax == 0 and scale == 1 and np.all(q == 0)
    # negative zeros keep their sign bit
    q, _, _ = oracle.quantize_pertensor(-z)
    assert np.all(q == 0x80)
    # NaN is ignored by amax and encodes to 0x7F
    x = np.array([np.nan, 1.0, -4.0], dtype=np.float32)
    q, amax, scale = oracle.quantize_pertensor(x)
    # qscale = 112: 1 -> 112 = 1.75 * 2^6 -> 0x6E, -4 -> -448 -> 0xFE
    assert amax == 4.0 and q.tolist() == [0x7F, 0x6E, 0xFE]
    # empty tensor
    q, amax, scale = oracle.quantize_pertensor(np.zeros((0, 7), dtype=np.float32))
    assert q.shape == (0, 7) and amax == 0 and scale == 1
    # a tiny amax whose 448/amax overflows fp32 falls back to scale 1
    t = np.array([1e-39, -5e-40], dtype=np.float32)
    q, amax, scale = oracle.quantize_pertensor(t)
    assert scale == 1 and np.all(q & 0x7F == 0)
    # an infinite element: qscale = 0, finite * 0 = 0, inf * 0 = NaN
    x = np.array([np.inf, 2.0, -3.0], dtype=np.float32)
    q, amax, scale = oracle.quantize_pertensor(x)
    assert np.isinf(amax) and np.isinf(scale) and q.tolist() == [0x7F, 0x00, 0x80]


def test_blockwise_tiles_are_independent_pertensor():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((70, 100)).astype(np.float32)
    x[5, 7] = 900.0
    q, s = oracle.quantize_blockwise_32x32(x)
    assert s.shape == (3, 4)
    for i in range(3):
        for j in range(4):
            blk = x[32 * i:32 * i + 32, 32 * j:32 * j + 32]
            qt, amax, st = oracle.quantize_pertensor(blk)
            assert st == s[i, j]
            assert np.array_equal(q[32 * i:32 * i + 32, 32 * j:32 * j + 32], qt)
            # the block's own amax maps to 448
            assert s[i, j] == np.float32(np.abs(blk).max()) / np.float32(448)
    # the outlier only affects its own tile
    assert s[0, 0] == np.float32(900.0) / np.float32(448.0)
    assert s[0, 1] < s[0, 0] / 50
