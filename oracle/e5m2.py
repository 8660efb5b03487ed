"""E5M2 (float8 e5m2) decode and round-to-nearest-even saturating encode.

[P3] (5th-gen tensor core paragraph, "Blackwell GPU 的核心创新") names the two
FP8 formats, E4M3 and E5M2.  E5M2 as [FP8] defines it: one sign bit s, a
5-bit exponent field e with bias 15, a 2-bit mantissa field m, following
IEEE-754 conventions:

  e == 0           : (-1)^s * (m/4) * 2^-14         (zero and subnormals)
  e == 31, m == 0  : (-1)^s * infinity
  e == 31, m != 0  : NaN
  otherwise        : (-1)^s * (1 + m/4) * 2^(e-15)

The largest finite magnitude is 0x7B = 1.75 * 2^15 = 57344.

The encoder saturates like the E4M3 one ("satfinite"): finite results only,
|x| > 57344 and +-infinity go to +-57344; NaN goes to 0x7F.
"""

import numpy as np

E5M2_MAX = 57344.0
NAN_CODE = 0x7F
MAX_CODE = 0x7B


def decode_code(c):
    """Value of one E5M2 code (an int in 0..255) as a Python float (exact)."""
    c = int(c)
    if not 0 <= c <= 255:
        raise ValueError("E5M2 code out of range")
    s = (c >> 7) & 1
    e = (c >> 2) & 0x1F
    m = c & 0x3
    sign = -1.0 if s else 1.0
    if e == 31:
        return sign * float("inf") if m == 0 else float("nan")
    if e == 0:
        return sign * (m / 4.0) * 2.0 ** -14
    return sign * (1.0 + m / 4.0) * 2.0 ** (e - 15)


_DECODE_TABLE = np.array([decode_code(c) for c in range(256)], dtype=np.float64)


def decode(codes):
    """Decode an array of E5M2 codes (uint8) to fp64 values, exactly."""
    codes = np.asarray(codes, dtype=np.uint8)
    return _DECODE_TABLE[codes]


# Non-negative finite magnitudes in code order, 0x00..0x7B (increasing).
_MAGS = _DECODE_TABLE[:MAX_CODE + 1].copy()
_MIDS = (_MAGS[:-1] + _MAGS[1:]) / 2.0    # exact: <= 4 significant bits


def encode(x):
    """Round fp32 values to E5M2 codes: nearest, ties to even, saturating.

    * NaN                          -> 0x7F
    * |x| > 57344 (incl. +-Inf)    -> sign | 0x7B
    * otherwise the nearest of the 124 non-negative finite magnitudes to |x|,
      a tie going to the code whose mantissa LSB is 0; the sign bit is copied
      from x.
    """
    x = np.asarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    sign = ((bits >> 31) & 1).astype(np.uint8) << 7
    ax = np.abs(x.astype(np.float64))
    isnan = np.isnan(ax)
    ax_safe = np.where(isnan, 0.0, ax)
    lo = np.searchsorted(_MAGS, ax_safe, side="right") - 1
    lo = np.clip(lo, 0, MAX_CODE)
    hi = np.minimum(lo + 1, MAX_CODE)
    mid = _MIDS[np.minimum(lo, MAX_CODE - 1)]
    exact = _MAGS[lo] == ax_safe
    below = ax_safe < mid
    above = ax_safe > mid
    tie_pick = np.where((lo & 1) == 0, lo, hi)
    mag = np.where(exact | below, lo, np.where(above, hi, tie_pick))
    mag = np.where(ax_safe > E5M2_MAX, MAX_CODE, mag)
    code = (mag.astype(np.uint8) | sign).astype(np.uint8)
    code = np.where(isnan, np.uint8(NAN_CODE), code).astype(np.uint8)
    return code.reshape(x.shape)
