"""CPU oracle for the FP8 E4M3 quantize + scaled GEMM path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this
package; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may use it.  It shares no code, table or helper with the
CUDA path under ``precision_linear_algebra_gb300/csrc``.

Everything here is plain numpy, written for a reader to check against the
definitions by eye: no blocking, no fusion, no reordering beyond what each
definition states.  Floating-point values are carried in fp64 wherever the
method does not fix the precision; where the method fixes fp32 (the amax, the
two scale divisions, the pre-cast multiply) numpy float32 arithmetic is used,
which is IEEE-754 binary32 with round-to-nearest-even.

Sources cited in the docstrings (the three web pages this method comes from):

[P1] "通过 CUTLASS 命名约定在 Triton 中实现 FP8 GEMM 内核" (blog.hotdry.top,
     2025-10-03): FP8 GEMM in Triton.  Body paragraphs: intro, Triton/CUTLASS
     tiles, evidence, kernel code, scale application ("此内核借鉴 CUTLASS"),
     optimisation parameter list ("优化参数清单"), monitoring ("监控要点"),
     risks ("风险考虑"), conclusion.
[P2] "利用 Cutlass 内核命名惯例在 Triton 中实现 FP8 张量核的多头注意力
     100 TFLOPS 加速": FP8 multi-head attention in Triton.
[P3] "JAX 中使用 Triton 优化 Blackwell GPU 的 FP8 GEMM 内核：TMA 异步加载与
     Warp 级原语" (blog.hotdry.top, 2025-10-07): FP8 GEMM for Blackwell.  Body
     paragraphs: intro, 5th-gen tensor cores ("Blackwell GPU 的核心创新"),
     warp specialisation ("Warp 级原语"), implementation and MoE
     ("要落地这些优化"), monitoring, checklist, conclusion.
[FP8] Micikevicius et al., "FP8 Formats for Deep Learning" (2022): the E4M3
     encoding that [P1] calls ``float8e4m3fn`` (bias 7, no infinities, a
     single NaN mantissa pattern, max 448), and E5M2 (bias 15, IEEE-style
     infinities and NaNs, max 57344), the second format [P3] names.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against facts that do not come from this code (the format's fixed values,
library casts, exact rational arithmetic, closed forms and invariants).
No function is "parity unpinned".
"""

from .e4m3 import decode_code, decode, encode, E4M3_MAX, NAN_CODE
from . import e5m2
from .bf16 import bf16_rne, bf16_bits_to_float
from .quantize import (amax_fp32, scales_from_amax, quantize_pertensor,
                       quantize_pertensor_delayed, quantize_blockwise_32x32,
                       quantize_pertensor_grouped)
from .gemm import (gemm_pertensor, gemm_blockscaled_32x32, gemm_grouped,
                   bound_pertensor, bound_blockscaled_32x32, max_abs_decoded,
                   max_abs_tile_scaled_32x32, tolerance_pertensor,
                   tolerance_blockscaled_32x32)

__all__ = [
    "decode_code", "decode", "encode", "E4M3_MAX", "NAN_CODE", "e5m2",
    "bf16_rne", "bf16_bits_to_float",
    "amax_fp32", "scales_from_amax", "quantize_pertensor",
    "quantize_blockwise_32x32", "quantize_pertensor_grouped",
    "gemm_pertensor", "gemm_blockscaled_32x32", "gemm_grouped",
    "bound_pertensor", "bound_blockscaled_32x32", "max_abs_decoded",
    "max_abs_tile_scaled_32x32", "tolerance_pertensor",
    "tolerance_blockscaled_32x32",
]
