"""E4M3 (float8 e4m3fn) decode and round-to-nearest-even saturating encode.

Format, as [FP8] defines it and as [P1] uses it ("输入 FP8E4M3（e4m3fn）",
optimisation parameter list; "E4M3: ±448", risks paragraph): one sign bit s,
a 4-bit exponent field e with bias 7, a 3-bit mantissa field m.

  e == 0           : (-1)^s * (m/8) * 2^-6          (zero and subnormals)
  e == 15, m == 7  : NaN                             (S.1111.111)
  otherwise        : (-1)^s * (1 + m/8) * 2^(e-7)

There is no infinity; the largest finite magnitude is 0x7E = 1.75 * 2^8 = 448.
"""

import numpy as np

E4M3_MAX = 448.0
NAN_CODE = 0x7F


def decode_code(c):
    """Value of one E4M3 code (an int in 0..255) as a Python float (exact)."""
    c = int(c)
    if not 0 <= c <= 255:
        raise ValueError("E4M3 code out of range")
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    sign = -1.0 if s else 1.0
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# All 256 values, built from the closed form above (fp64 holds every one exactly).
_DECODE_TABLE = np.array([decode_code(c) for c in range(256)], dtype=np.float64)


def decode(codes):
    """Decode an array of E4M3 codes (uint8) to fp64 values, exactly."""
    codes = np.asarray(codes, dtype=np.uint8)
    return _DECODE_TABLE[codes]


# Non-negative finite magnitudes in code order: codes 0x00..0x7E are increasing.
_MAGS = _DECODE_TABLE[:0x7F].copy()
# Midpoint between neighbouring magnitudes.  Each magnitude has at most four
# significant bits, so the midpoint is exact in fp64.
_MIDS = (_MAGS[:-1] + _MAGS[1:]) / 2.0


def encode(x):
    """Round fp32 values to E4M3 codes: nearest, ties to even, saturating.

    * NaN                        -> 0x7F
    * |x| > 448 (incl. +-Inf)    -> sign | 0x7E      (saturate, "satfinite")
    * otherwise the nearest of the 127 non-negative finite magnitudes to |x|,
      a tie going to the code whose mantissa LSB is 0; the sign bit is copied
      from x, so -0.0 and negatives that round to zero give 0x80.

    Distances are decided by comparing |x| with the exact midpoint between
    the two neighbouring magnitudes, so no subtraction rounds.
    """
    x = np.asarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    sign = ((bits >> 31) & 1).astype(np.uint8) << 7
    ax = np.abs(x.astype(np.float64))
    isnan = np.isnan(ax)
    ax_safe = np.where(isnan, 0.0, ax)

    # lo = largest code whose magnitude is <= |x| (clipped to the finite range).
    lo = np.searchsorted(_MAGS, ax_safe, side="right") - 1
    lo = np.clip(lo, 0, 0x7E)
    hi = np.minimum(lo + 1, 0x7E)
    mid = _MIDS[np.minimum(lo, 0x7D)]
    exact = _MAGS[lo] == ax_safe
    below = ax_safe < mid
    above = ax_safe > mid
    tie_pick = np.where((lo & 1) == 0, lo, hi)
    mag = np.where(exact | below, lo, np.where(above, hi, tie_pick))
    mag = np.where(ax_safe > E4M3_MAX, 0x7E, mag)
    code = (mag.astype(np.uint8) | sign).astype(np.uint8)
    code = np.where(isnan, np.uint8(NAN_CODE), code).astype(np.uint8)
    return code.reshape(x.shape)
