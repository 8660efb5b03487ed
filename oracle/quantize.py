"""Per-tensor and 32x32 block amax -> scale -> E4M3 quantisation.

[P1] (risks paragraph) states that E4M3's range is +-448 and that per-tensor
scaling is needed to avoid overflow ("需 per-tensor 缩放避免溢出"), and the
parameter list fixes the threshold "scale_max=448".  [P3] (implementation
paragraph) sets the scale granularity to 32x32 blocks ("缩放粒度为 32x32 块").

The steps, in the order the method takes them:

1. amax = max_i |x_i| over the tensor (or tile), NaN ignored, in fp32.
   Max is exact, so the order of the reduction does not matter.
2. qscale = fp32(448 / amax), the multiplier applied before the cast, and
   scale  = fp32(amax / 448), the dequantisation factor the GEMM consumes
   (57344 in place of 448 for the E5M2 variant).
   Both are single IEEE fp32 divisions; neither is derived from the other.
   If amax == 0 or qscale is not finite, qscale = scale = 1.
3. q_i = E4M3_RNE_satfinite(fp32(x_i * qscale)): one fp32 multiply, then the
   saturating round-to-nearest-even encode.

Delayed scaling (``quantize_pertensor_delayed``) is a reading of ours, not a
step the pages describe: it takes steps 2 and 3 with an amax carried over
from an earlier call (the previous training or inference step) in place of
step 1's, and performs step 1 on the current tensor only to record its amax
for the next call.  The pages' remark that per-tensor scaling keeps values
inside E4M3's +-448 then holds only up to the saturation of step 3: values
beyond the carried-over amax land on the largest code.
"""

import numpy as np

from . import e4m3, e5m2

# format -> (largest finite magnitude, saturating RNE encoder)
FORMATS = {"e4m3": (e4m3.E4M3_MAX, e4m3.encode),
           "e5m2": (e5m2.E5M2_MAX, e5m2.encode)}


def amax_fp32(x):
    """max |x| over all elements, NaN ignored, as an fp32 scalar (0 if none)."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).reshape(-1)
    a = a[~np.isnan(a)]
    if a.size == 0:
        return np.float32(0.0)
    return np.float32(a.max())


def scales_from_amax(amax, fmt="e4m3"):
    """(qscale, scale) as fp32 scalars, by the two IEEE fp32 divisions
    qscale = fmax / amax and scale = amax / fmax (fmax = 448 for E4M3, 57344
    for E5M2)."""
    amax = np.float32(amax)
    fmax = np.float32(FORMATS[fmt][0])
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        qscale = np.float32(fmax / amax)
        scale = np.float32(amax / fmax)
    if amax == 0 or not np.isfinite(qscale):
        return np.float32(1.0), np.float32(1.0)
    return qscale, scale


def quantize_pertensor(x, fmt="e4m3"):
    """Quantise an fp32 array with one per-tensor scale.

    Returns (codes uint8 with x's shape, amax fp32, scale fp32).  fmt is
    "e4m3" (the method's format) or "e5m2".
    """
    x = np.asarray(x, dtype=np.float32)
    amax = amax_fp32(x)
    qscale, scale = scales_from_amax(amax, fmt)
    with np.errstate(over="ignore", invalid="ignore"):
        y = (x * qscale).astype(np.float32)      # fp32 * fp32 -> fp32, RNE
    return FORMATS[fmt][1](y), amax, scale


def quantize_pertensor_delayed(x, amax_prev, fmt="e4m3"):
    """Quantise with the scale of a carried-over amax (delayed scaling).

    Steps 2 and 3 of the per-tensor scheme with ``amax_prev`` in place of the
    tensor's own amax; step 1 on x gives the amax recorded for the next call.
    Returns (codes uint8 with x's shape, amax of x fp32, scale fp32), where
    scale = fp32(amax_prev / fmax) is the dequantisation factor of the codes.
    """
    x = np.asarray(x, dtype=np.float32)
    qscale, scale = scales_from_amax(np.float32(amax_prev), fmt)
    with np.errstate(over="ignore", invalid="ignore"):
        y = (x * qscale).astype(np.float32)      # fp32 * fp32 -> fp32, RNE
    return FORMATS[fmt][1](y), amax_fp32(x), scale


def quantize_blockwise_32x32(x):
    """Quantise a 2-D fp32 array with one scale per 32x32 tile.

    Tile (i, j) covers rows 32i..32i+31 and columns 32j..32j+31, cut short at
    the array's edge (ragged edge tiles use their actual extent).  Each tile is
    quantised exactly as ``quantize_pertensor`` quantises a whole tensor.

    Returns (codes uint8 [R][C], scales fp32 [ceil(R/32)][ceil(C/32)]).
    """
    x = np.asarray(x, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError("expected a 2-D array")
    R, C = x.shape
    tr, tc = -(-R // 32), -(-C // 32)
    codes = np.empty((R, C), dtype=np.uint8)
    scales = np.empty((tr, tc), dtype=np.float32)
    for i in range(tr):
        for j in range(tc):
            rs = slice(32 * i, min(32 * i + 32, R))
            cs = slice(32 * j, min(32 * j + 32, C))
            q, _, s = quantize_pertensor(x[rs, cs])
            codes[rs, cs] = q
            scales[i, j] = s
    return codes, scales


def quantize_pertensor_grouped(x, m_offsets):
    """Per-tensor quantisation of each row group of a 2-D fp32 array.

    Group e is rows m_offsets[e] .. m_offsets[e+1]-1 of x (one MoE expert's
    tokens, [P3] implementation paragraph: the grouped GEMM for MoE), and is
    quantised exactly as ``quantize_pertensor`` quantises a whole tensor,
    with its own amax and scale; a group with no rows has amax 0 and scale 1
    (steps 1 and 2 on an empty tensor).  Rows at or past m_offsets[E] belong
    to no group.

    Returns (codes uint8 [m_offsets[E]][C], amax fp32 [E], scale fp32 [E]).
    """
    x = np.asarray(x, dtype=np.float32)
    offs = [int(v) for v in m_offsets]
    E = len(offs) - 1
    if x.ndim != 2 or offs[0] != 0 or any(b < a for a, b in zip(offs, offs[1:])) \
            or offs[-1] > x.shape[0]:
        raise ValueError("m_offsets must start at 0, not decrease and fit the rows of x")
    codes = np.empty((offs[-1], x.shape[1]), dtype=np.uint8)
    amax = np.empty(E, dtype=np.float32)
    scale = np.empty(E, dtype=np.float32)
    for e in range(E):
        q, amax[e], scale[e] = quantize_pertensor(x[offs[e]:offs[e + 1]])
        codes[offs[e]:offs[e + 1]] = q
    return codes, amax, scale

