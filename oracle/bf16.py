"""Round fp64 values directly to bfloat16, round-to-nearest-even.

BF16 is the GEMM output type ([P1], optimisation parameter list: "累加器
FP32，输出 dequantize 回 BF16").  bfloat16 has a sign bit, an 8-bit exponent
with bias 127 and 7 stored mantissa bits (8 significant bits).  Normal values
have magnitude in [2^-126, (2 - 2^-7) * 2^127]; subnormals are multiples of
2^-133.  The rounding here goes straight from fp64 to bf16 (one rounding),
never through fp32 (which would round twice).
"""

import numpy as np


def bf16_rne(r):
    """Round an fp64 array to bf16; return the uint16 bit patterns.

    For a finite r != 0 let E be the exponent of its leading bit
    (2^E <= |r| < 2^(E+1)).  The bf16 quantum there is q = 2^(E-7), but not
    below the subnormal quantum 2^-133.  |r|/q is rounded to an integer with
    ties to even (numpy.rint), and multiplied back.  A result of 2^128 or more
    is an overflow and becomes infinity.  The sign is copied from r, so
    values that round to zero keep their sign.  NaN maps to 0x7FC0.
    """
    r = np.asarray(r, dtype=np.float64)
    out_shape = r.shape
    r = r.reshape(-1)
    ar = np.abs(r)
    finite_nz = np.isfinite(ar) & (ar != 0.0)
    safe = np.where(finite_nz, ar, 1.0)
    _, e_plus_1 = np.frexp(safe)            # safe = m * 2^e_plus_1, m in [0.5, 1)
    lead = e_plus_1.astype(np.int64) - 1    # exponent of the leading bit
    qexp = np.maximum(lead - 7, -133)
    n = np.ldexp(safe, -qexp)               # exact: scaling by a power of two
    n = np.rint(n)                          # ties to even
    mag = np.ldexp(n, qexp)
    mag = np.where(mag >= 2.0 ** 128, np.inf, mag)
    mag = np.where(finite_nz, mag, ar)      # 0, inf and nan pass through
    val = np.copysign(mag, r)
    # Every value in val is now exactly representable in bf16, hence in fp32,
    # so its fp32 bit pattern's top half is the bf16 pattern.
    bits = (val.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bits = np.where(np.isnan(r), np.uint16(0x7FC0), bits).astype(np.uint16)
    return bits.reshape(out_shape)


def bf16_bits_to_float(bits):
    """bf16 bit patterns (uint16) to fp64 values, exactly."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
