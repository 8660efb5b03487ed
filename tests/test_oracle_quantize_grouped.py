"""Pins for the oracle's grouped per-tensor quantiser (CPU only).

Group e (rows m_offsets[e] .. m_offsets[e+1]-1) is quantised as one tensor
with its own amax ([P3] implementation paragraph: the MoE grouped GEMM;
[P1] risks paragraph: per-tensor scaling).  Pins:

* a hand-worked example, codes written out from the E4M3 encoding ([FP8]:
  bias 7, 3 mantissa bits, 0x7E = 448, 0x7F = NaN), including an empty group
  (amax 0, scale 1), a NaN (ignored by the amax, code 0x7F) and a product
  that rounds to the largest code;
* reductions: one group is the per-tensor quantiser; groups of independent
  tensors are the per-tensor quantiser on each;
* planted mistakes (a group boundary one row off, one amax for all groups,
  the neighbour's scale for an empty group) fail the hand example.
"""

import numpy as np
import pytest

import oracle

NAN = np.float32("nan")
X = np.array([[1.5, -3.0],
              [0.25, 2.0],
              [0.0, -0.5],
              [1000.0, 7.0],
              [NAN, 1.0]], dtype=np.float32)
OFFS = [0, 2, 2, 5]

# group 0: amax 3, qscale = fp32(448/3):
#   1.5 -> 224 = 1.75 * 2^7        -> 0 1110 110 = 0x76
#  -3.0 -> 448 (largest)           -> 1 1111 110 = 0xFE
#   0.25 -> 37.33, nearest 36 = 1.125 * 2^5 -> 0 1100 001 = 0x61
#   2.0 -> 298.67, nearest 288 = 1.125 * 2^8 -> 0 1111 001 = 0x79
# group 1: no rows -> amax 0, scale 1
# group 2: amax 1000 (NaN ignored), qscale = fp32(0.448):
#   0.0 -> 0x00;  -0.5 -> -0.224 = -1.792 * 2^-3, nearest -1.75 * 2^-3 -> 1 0100 110 = 0xA6
#   1000 -> 448.00001 -> 448       -> 0 1111 110 = 0x7E
#   7.0 -> 3.136 = 1.568 * 2, nearest 1.625 * 2 -> 0 1000 101 = 0x45
#   NaN -> 0x7F;  1.0 -> 0.448 = 1.792 * 2^-2, nearest 1.75 * 2^-2 -> 0 0101 110 = 0x2E
CODES = np.array([[0x76, 0xFE],
                  [0x61, 0x79],
                  [0x00, 0xA6],
                  [0x7E, 0x45],
                  [0x7F, 0x2E]], dtype=np.uint8)
AMAX = np.array([3.0, 0.0, 1000.0], dtype=np.float32)
SCALE = np.array([np.float32(3.0) / np.float32(448.0), 1.0,
                  np.float32(1000.0) / np.float32(448.0)], dtype=np.float32)


def _matches(fn):
    q, amax, scale = fn(X, OFFS)
    return (np.array_equal(q, CODES) and np.array_equal(amax, AMAX)
            and np.array_equal(scale, SCALE))


def test_hand_example():
    assert _matches(oracle.quantize_pertensor_grouped)


def test_one_group_is_the_per_tensor_quantiser():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((37, 19)) * 5).astype(np.float32)
    q, amax, scale = oracle.quantize_pertensor_grouped(x, [0, 37])
    rq, ra, rs = oracle.quantize_pertensor(x)
    assert np.array_equal(q, rq) and amax[0] == ra and scale[0] == rs


def test_groups_of_independent_tensors():
    rng = np.random.default_rng(5)
    parts = [(rng.standard_normal((n, 24)) * 10.0 ** p).astype(np.float32)
             for n, p in ((3, -4), (0, 0), (50, 2), (1, 6), (12, 0))]
    offs = np.concatenate([[0], np.cumsum([p.shape[0] for p in parts])])
    x = np.concatenate(parts + [np.full((4, 24), 1e30, np.float32)])  # rows past the groups
    q, amax, scale = oracle.quantize_pertensor_grouped(x, offs)
    assert q.shape == (offs[-1], 24)
    for e, p in enumerate(parts):
        rq, ra, rs = oracle.quantize_pertensor(p)
        assert np.array_equal(q[offs[e]:offs[e + 1]], rq)
        assert amax[e] == ra and scale[e] == rs


def test_bad_offsets_are_rejected():
    for offs in ([1, 5], [0, 3, 2], [0, 6]):
        with pytest.raises(ValueError):
            oracle.quantize_pertensor_grouped(X, offs)


# ------------------------------------------------------------ planted mistakes
def _boundary_off_by_one(x, m_offsets):
    # the inner boundaries one row early (still valid offsets)
    offs = [int(v) for v in m_offsets]
    offs = [offs[0]] + [max(v - 1, 0) for v in offs[1:-1]] + [offs[-1]]
    return oracle.quantize_pertensor_grouped(x, offs)


def _one_amax_for_all(x, m_offsets):
    offs = [int(v) for v in m_offsets]
    _, a, s = oracle.quantize_pertensor(x[:offs[-1]])
    q, _, _ = oracle.quantize_pertensor(x[:offs[-1]])
    E = len(offs) - 1
    return q, np.full(E, a, np.float32), np.full(E, s, np.float32)


def _empty_group_takes_neighbour(x, m_offsets):
    q, amax, scale = oracle.quantize_pertensor_grouped(x, m_offsets)
    for e in range(len(amax)):
        if m_offsets[e + 1] == m_offsets[e] and e > 0:
            amax[e], scale[e] = amax[e - 1], scale[e - 1]
    return q, amax, scale


@pytest.mark.parametrize("mutant", [_boundary_off_by_one, _one_amax_for_all,
                                    _empty_group_takes_neighbour])
def test_planted_mistakes_fail_the_hand_example(mutant):
    assert not _matches(mutant)
