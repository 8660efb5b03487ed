"""GB300 (sm_103a) FP8 E4M3 quantize + scaled GEMM library: Python binding.

The compute lives in ``libfp8la.so`` (CUDA C++ with inline PTX, built from
``csrc/`` by ``build.py``); its C ABI is ``include/fp8la.h``.  This module
only marshals arguments: it loads the library with ctypes, exposes each C
entry point under the same name (``fp8_quantize_pertensor``, ``fp8_gemm``,
``fp8_gemm_blockscaled_32x32``, ``fp8_grouped_gemm``, ...) taking raw
integers for pointers, and adds thin torch-tensor wrappers (``quantize_*``,
``gemm*``) that allocate outputs with torch and pass ``data_ptr()`` and the
current CUDA stream.  There is no fallback: if the library cannot be loaded
or a call fails, an exception is raised.
"""

import ctypes
import os

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libfp8la.so")

FP8LA_OK = 0
FP8LA_ERR_INVALID_ARG = -1
FP8LA_ERR_ALIGNMENT = -2
FP8LA_ERR_UNSUPPORTED = -3
FP8LA_ERR_CUDA = -4
FP8LA_ERR_DEVICE_TIMEOUT = -5
FP8LA_ERR_DEVICE_ARG = -6
FP8LA_FORMAT_E4M3 = 0
FP8LA_FORMAT_E5M2 = 1
_FORMATS = {"e4m3": FP8LA_FORMAT_E4M3, "e5m2": FP8LA_FORMAT_E5M2}

# (name, restype, argtypes) of every entry point in include/fp8la.h.
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_S = ctypes.c_int
SIGNATURES = [
    ("fp8_quantize_pertensor", _S, [_P, _I64, _I64, _I64, _P, _I64, _P, _P, _P]),
    ("fp8_quantize_pertensor_ex", _S, [_P, _I64, _I64, _I64, _P, _I64, _P, _P, _I32, _P]),
    ("fp8_quantize_pertensor_delayed", _S,
     [_P, _I64, _I64, _I64, _P, _I64, _P, _P, _P, _I32, _P]),
    ("fp8_quantize_blockwise_32x32", _S, [_P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P]),
    ("fp8_quantize_pertensor_grouped", _S,
     [_P, _I32, _P, _I64, _I64, _I64, _P, _I64, _P, _P, _P]),
    ("fp8_gemm", _S, [_P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I64, _P, _P, _P]),
    ("fp8_gemm_ex", _S, [_P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I64, _P, _P, _I32, _I32, _P]),
    ("fp8_gemm_blockscaled_32x32", _S,
     [_P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I64, _P, _I64, _P, _I64, _P]),
    ("fp8_grouped_gemm", _S,
     [_I32, _P, _I64, _P, _I64, _P, _I64, _I64, _P, _I64, _I64, _I64, _P, _P, _P]),
    ("fp8_get_device_status", _S, [_P]),
    ("fp8la_set_wait_timeout_ns", _S, [_I64]),
    ("fp8la_diag_gemm_withheld_arrival", _S, [_P, _I64, _P, _I64, _P, _I64, _P, _P, _P]),
    ("fp8la_diag_withheld_arrival", _S,
     [_I32, _P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I64, _P, _I64, _P, _I64, _P]),
    ("fp8la_set_gemm_variant", _S, [_I32]),
    ("fp8la_status_string", ctypes.c_char_p, [_S]),
    ("fp8la_version", _S, []),
]

_lib = None


class Fp8laError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (what, status_string(status), status))


def load(path=None):
    """Load libfp8la.so (build it first with build.build()); raise if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            "libfp8la.so is not built (%s); run `python -m "
            "precision_linear_algebra_gb300.build`" % p)
    lib = ctypes.CDLL(p)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def status_string(status):
    try:
        return load().fp8la_status_string(status).decode()
    except Exception:
        return "status %d" % status


def _call(name, *args):
    st = getattr(load(), name)(*args)
    if st != FP8LA_OK:
        raise Fp8laError(st, name)
    return st


# --------------------------------------------------- raw C-ABI entry points
def fp8_quantize_pertensor(x, rows, cols, ldx, q, ldq, amax_out, scale_out, stream):
    return _call("fp8_quantize_pertensor", x, rows, cols, ldx, q, ldq, amax_out,
                 scale_out, stream)


def fp8_quantize_pertensor_delayed(x, rows, cols, ldx, q, ldq, amax_prev, amax_out, scale_out,
                                   fmt, stream):
    return _call("fp8_quantize_pertensor_delayed", x, rows, cols, ldx, q, ldq, amax_prev,
                 amax_out, scale_out, fmt, stream)


def fp8_quantize_pertensor_ex(x, rows, cols, ldx, q, ldq, amax_out, scale_out, fmt, stream):
    return _call("fp8_quantize_pertensor_ex", x, rows, cols, ldx, q, ldq, amax_out,
                 scale_out, fmt, stream)


def fp8_gemm_ex(A, lda, B, ldb, C, ldc, M, N, K, scale_a, scale_b, a_fmt, b_fmt, stream):
    return _call("fp8_gemm_ex", A, lda, B, ldb, C, ldc, M, N, K, scale_a, scale_b,
                 a_fmt, b_fmt, stream)


def fp8_quantize_blockwise_32x32(x, rows, cols, ldx, q, ldq, scales, ld_scales, stream):
    return _call("fp8_quantize_blockwise_32x32", x, rows, cols, ldx, q, ldq,
                 scales, ld_scales, stream)


def fp8_quantize_pertensor_grouped(x, num_groups, m_offsets, rows_capacity, cols, ldx, q, ldq,
                                   amax_out, scale_out, stream):
    return _call("fp8_quantize_pertensor_grouped", x, num_groups, m_offsets, rows_capacity,
                 cols, ldx, q, ldq, amax_out, scale_out, stream)


def fp8_gemm(A, lda, B, ldb, C, ldc, M, N, K, scale_a, scale_b, stream):
    return _call("fp8_gemm", A, lda, B, ldb, C, ldc, M, N, K, scale_a, scale_b, stream)


def fp8_gemm_blockscaled_32x32(A, lda, B, ldb, C, ldc, M, N, K, sa, ld_sa, sb,
                               ld_sb, stream):
    return _call("fp8_gemm_blockscaled_32x32", A, lda, B, ldb, C, ldc, M, N, K,
                 sa, ld_sa, sb, ld_sb, stream)


def fp8_grouped_gemm(num_groups, m_offsets, m_capacity, A, lda, B, ldb,
                     b_group_stride, C, ldc, N, K, scale_a, scale_b, stream):
    return _call("fp8_grouped_gemm", num_groups, m_offsets, m_capacity, A, lda,
                 B, ldb, b_group_stride, C, ldc, N, K, scale_a, scale_b, stream)


def fp8_get_device_status(stream):
    """Sync `stream`, read and clear the device status word; return it."""
    return load().fp8_get_device_status(stream)


def fp8la_set_wait_timeout_ns(ns):
    return _call("fp8la_set_wait_timeout_ns", int(ns))


def fp8la_diag_gemm_withheld_arrival(A, lda, B, ldb, C, ldc, scale_a, scale_b, stream):
    return _call("fp8la_diag_gemm_withheld_arrival", A, lda, B, ldb, C, ldc,
                 scale_a, scale_b, stream)


FP8LA_DIAG_KERNEL_PAIR = 1
FP8LA_DIAG_KERNEL_BLOCK32 = 2


def fp8la_diag_withheld_arrival(kernel, A, lda, B, ldb, C, ldc, M, N, K, scale_a, ld_sa,
                                scale_b, ld_sb, stream):
    return _call("fp8la_diag_withheld_arrival", kernel, A, lda, B, ldb, C, ldc, M, N, K,
                 scale_a, ld_sa, scale_b, ld_sb, stream)


def fp8la_set_gemm_variant(variant):
    """0 = by shape, 1 = single-CTA kernel, 2 = CTA-pair kernel, 3 = single-CTA
    kernel with 128 x 128 tiles, 4 = two CTA pairs per cluster sharing A."""
    return _call("fp8la_set_gemm_variant", int(variant))


def fp8la_version():
    return load().fp8la_version()


# ------------------------------------------------------ torch conveniences
def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def _ptr(t):
    return t.data_ptr() if t is not None else None


def _ld(t):
    """Leading dimension of a row-major 2-D tensor.  A single-row tensor's
    row stride is meaningless (torch keeps whatever it was given, even 0), so
    its row length is used."""
    return t.stride(0) if t.shape[0] > 1 else max(t.shape[1], 1)


def _ld_tma(t):
    """As _ld, for an FP8 GEMM operand, whose row stride goes into a TMA
    descriptor (a multiple of 16 bytes even when there is one row: the
    stride of a single row never addresses memory, so the row length
    rounded up to 16 is passed)."""
    return t.stride(0) if t.shape[0] > 1 else (max(t.shape[1], 1) + 15) // 16 * 16


def _ld_scales(t):
    """As _ld, for a block-scale grid, whose row stride the GEMM reads by TMA
    (a multiple of 4 floats even when there is one row)."""
    return t.stride(0) if t.shape[0] > 1 else (t.shape[1] + 3) // 4 * 4


def quantize_pertensor(x, q=None, amax=None, scale=None, fmt="e4m3"):
    """x: fp32 CUDA [rows][cols] (row stride may exceed cols).

    Returns (q uint8 [rows][cols], amax fp32 [1], scale fp32 [1]), all on
    x's device; nothing is synchronised.  fmt: "e4m3" or "e5m2".
    """
    import torch
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    amax = torch.empty(1, dtype=torch.float32, device=x.device) if amax is None else amax
    scale = torch.empty(1, dtype=torch.float32, device=x.device) if scale is None else scale
    fp8_quantize_pertensor_ex(_ptr(x), rows, cols, _ld(x), _ptr(q), _ld(q),
                              _ptr(amax), _ptr(scale), _FORMATS[fmt], _stream())
    return q, amax, scale


def quantize_pertensor_delayed(x, amax_prev, q=None, amax=None, scale=None, fmt="e4m3"):
    """One-pass quantisation with the scale of a carried-over amax.

    x: fp32 CUDA [rows][cols]; amax_prev: fp32 CUDA tensor holding one value
    (e.g. the amax this call returned at the previous step).  Returns
    (q uint8 [rows][cols], amax fp32 [1] of x, scale fp32 [1] of the codes);
    amax must not share storage with amax_prev.
    """
    import torch
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    amax = torch.empty(1, dtype=torch.float32, device=x.device) if amax is None else amax
    scale = torch.empty(1, dtype=torch.float32, device=x.device) if scale is None else scale
    fp8_quantize_pertensor_delayed(_ptr(x), rows, cols, _ld(x), _ptr(q), _ld(q),
                                   _ptr(amax_prev), _ptr(amax), _ptr(scale),
                                   _FORMATS[fmt], _stream())
    return q, amax, scale


def quantize_blockwise_32x32(x, q=None, scales=None):
    """x: fp32 CUDA [rows][cols] -> (q uint8, scales fp32 [ceil(r/32)][ceil(c/32)])."""
    import torch
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if scales is None:
        # leading dimension rounded up to 4 floats, as the block-scaled GEMM
        # reads scale grids with TMA (16-byte rows)
        tc = (cols + 31) // 32
        scales = torch.empty(((rows + 31) // 32, (tc + 3) // 4 * 4),
                             dtype=torch.float32, device=x.device)[:, :tc]
    fp8_quantize_blockwise_32x32(_ptr(x), rows, cols, _ld(x), _ptr(q), _ld(q),
                                 _ptr(scales), _ld(scales), _stream())
    return q, scales


def quantize_pertensor_grouped(x, m_offsets, q=None, amax=None, scale=None):
    """x: fp32 CUDA [rows_capacity][cols]; m_offsets: int32 CUDA [E+1].

    Group e (rows m_offsets[e] .. m_offsets[e+1]-1) is quantised with its own
    per-tensor amax and scale.  Returns (q uint8 [rows_capacity][cols],
    amax fp32 [E], scale fp32 [E]); nothing is synchronised.
    """
    import torch
    assert x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1
    assert m_offsets.dtype == torch.int32 and m_offsets.dim() == 1
    rows, cols = x.shape
    E = m_offsets.numel() - 1
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    amax = torch.empty(E, dtype=torch.float32, device=x.device) if amax is None else amax
    scale = torch.empty(E, dtype=torch.float32, device=x.device) if scale is None else scale
    fp8_quantize_pertensor_grouped(_ptr(x), E, _ptr(m_offsets), rows, cols, _ld(x), _ptr(q),
                                   _ld(q), _ptr(amax), _ptr(scale), _stream())
    return q, amax, scale


def gemm(A, B, scale_a, scale_b, C=None, a_fmt="e4m3", b_fmt="e4m3"):
    """A uint8 [M][K], B uint8 [N][K] (K-major), scales fp32 [1] -> C bf16 [M][N].

    a_fmt, b_fmt: "e4m3" (default, fp8_gemm) or "e5m2" (fp8_gemm_ex)."""
    import torch
    M, K = A.shape
    N = B.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if a_fmt == "e4m3" and b_fmt == "e4m3":
        fp8_gemm(_ptr(A), _ld_tma(A), _ptr(B), _ld_tma(B), _ptr(C), _ld(C),
                 M, N, K, _ptr(scale_a), _ptr(scale_b), _stream())
    else:
        fp8_gemm_ex(_ptr(A), _ld_tma(A), _ptr(B), _ld_tma(B), _ptr(C), _ld(C),
                    M, N, K, _ptr(scale_a), _ptr(scale_b), _FORMATS[a_fmt],
                    _FORMATS[b_fmt], _stream())
    return C


def gemm_blockscaled_32x32(A, B, sa, sb, C=None):
    """Block-scaled GEMM; sa [ceil(M/32)][ceil(K/32)], sb [ceil(N/32)][ceil(K/32)]."""
    import torch
    M, K = A.shape
    N = B.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    fp8_gemm_blockscaled_32x32(_ptr(A), _ld_tma(A), _ptr(B), _ld_tma(B), _ptr(C),
                               _ld(C), M, N, K, _ptr(sa), _ld_scales(sa),
                               _ptr(sb), _ld_scales(sb), _stream())
    return C


def grouped_gemm(m_offsets, A, B, scale_a, scale_b, C=None):
    """m_offsets int32 [E+1] (device); A [cap][K]; B [E][N][K]; scales [E]."""
    import torch
    E = B.shape[0]
    cap, K = A.shape
    N = B.shape[1]
    if C is None:
        C = torch.empty((cap, N), dtype=torch.bfloat16, device=A.device)
    ldb = B.stride(1) if N > 1 else (max(K, 1) + 15) // 16 * 16
    bstride = B.stride(0) if E > 1 else N * ldb
    fp8_grouped_gemm(E, _ptr(m_offsets), cap, _ptr(A), _ld_tma(A), _ptr(B),
                     ldb, bstride, _ptr(C), _ld(C), N, K,
                     _ptr(scale_a), _ptr(scale_b), _stream())
    return C


def device_status():
    return fp8_get_device_status(_stream())
