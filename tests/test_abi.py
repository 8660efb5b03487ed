"""CPU checks of the C ABI: the library builds, loads, exports every entry
point that include/*.h declares, and rejects bad arguments on the host
before touching the GPU.  No compute call is made here."""

import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*FP8LA_API\s+(?:const\s+)?\w+\s*\*?\s*(fp8\w*)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from precision_linear_algebra_gb300 import build
    import precision_linear_algebra_gb300 as fl
    build.build()
    return fl.load()


def test_header_declares_the_four_method_calls():
    names = _declared()
    for n in ["fp8_quantize_pertensor", "fp8_gemm", "fp8_gemm_blockscaled_32x32",
              "fp8_grouped_gemm"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    import precision_linear_algebra_gb300 as fl
    bound = {n for n, _, _ in fl.SIGNATURES}
    for name in _declared():
        assert hasattr(lib, name), name
        assert name in bound, "binding lacks " + name


def test_status_strings_and_version(lib):
    assert lib.fp8la_status_string(0) == b"FP8LA_OK"
    assert lib.fp8la_status_string(-5) == b"FP8LA_ERR_DEVICE_TIMEOUT"
    assert lib.fp8la_status_string(-6) == b"FP8LA_ERR_DEVICE_ARG"
    assert lib.fp8la_version() >= 100


def test_host_argument_rejection(lib):
    """Validation that runs before any CUDA call."""
    P = ctypes.c_void_p
    one = P(16)
    # quantize: NULL amax/scale, negative sizes, ld < cols
    assert lib.fp8_quantize_pertensor(one, 4, 4, 4, one, 4, None, one, None) == -1
    assert lib.fp8_quantize_pertensor(one, -1, 4, 4, one, 4, one, one, None) == -1
    assert lib.fp8_quantize_pertensor(one, 4, 8, 4, one, 8, one, one, None) == -1
    # amax_out and scale_out must be two different words
    two = P(32)
    assert lib.fp8_quantize_pertensor(one, 4, 4, 4, one, 4, two, two, None) == -1
    assert lib.fp8_quantize_pertensor_ex(one, 4, 4, 4, one, 4, two, two, 0, None) == -1
    assert lib.fp8_quantize_pertensor_ex(one, 0, 4, 4, one, 4, two, two, 1, None) == -1
    assert lib.fp8_quantize_blockwise_32x32(one, 4, 64, 64, one, 64, one, 1, None) == -1
    # delayed scaling: the carried-over amax, the new amax and the scale must
    # be three different words; bad format
    two, three = P(32), P(48)
    assert lib.fp8_quantize_pertensor_delayed(one, 4, 4, 4, one, 4, two, two, three, 0, None) == -1
    assert lib.fp8_quantize_pertensor_delayed(one, 4, 4, 4, one, 4, two, three, two, 0, None) == -1
    assert lib.fp8_quantize_pertensor_delayed(one, 4, 4, 4, one, 4, None, two, three, 0, None) == -1
    assert lib.fp8_quantize_pertensor_delayed(one, 4, 4, 4, one, 4, one, two, three, 7, None) == -1
    # gemm: negative sizes, ldc < N, lda < K, misaligned operands
    assert lib.fp8_gemm(one, 16, one, 16, one, 8, -1, 8, 16, one, one, None) == -1
    assert lib.fp8_gemm(one, 16, one, 16, one, 4, 8, 8, 16, one, one, None) == -1
    assert lib.fp8_gemm(one, 16, one, 32, one, 8, 8, 8, 32, one, one, None) == -1
    assert lib.fp8_gemm(P(17), 32, one, 32, one, 8, 8, 8, 32, one, one, None) == -2
    assert lib.fp8_gemm(one, 24, one, 32, one, 8, 8, 8, 24, one, one, None) == -2
    assert lib.fp8_gemm(one, 16, one, 16, P(33), 8, 8, 8, 16, one, one, None) == -2
    # M == 0 or N == 0 is a no-op that succeeds without touching the GPU
    assert lib.fp8_gemm(None, 16, None, 16, None, 8, 0, 8, 16, None, None, None) == 0
    assert lib.fp8_gemm(None, 16, None, 16, None, 8, 8, 0, 16, None, None, None) == 0
    # block-scaled: scale grids must allow 16-byte TMA rows
    assert lib.fp8_gemm_blockscaled_32x32(one, 64, one, 64, one, 64, 64, 64, 64,
                                          one, 2, one, 4, None) == -2
    assert lib.fp8_gemm_blockscaled_32x32(one, 64, one, 64, one, 64, 64, 64, 64,
                                          P(20), 4, one, 4, None) == -2
    assert lib.fp8_gemm_blockscaled_32x32(one, 64, one, 64, one, 64, 64, 64, 64,
                                          one, 1, one, 4, None) == -1
    # grouped: group count out of range, NULL offsets
    assert lib.fp8_grouped_gemm(0, one, 8, one, 16, one, 16, 256, one, 8, 8, 16, one, one, None) == -1
    assert lib.fp8_grouped_gemm(2000, one, 8, one, 16, one, 16, 256, one, 8, 8, 16, one, one, None) == -1
    assert lib.fp8_grouped_gemm(2, None, 8, one, 16, one, 16, 256, one, 8, 8, 16, one, one, None) == -1
    # grouped quantiser: group count out of range, NULL offsets, ld < cols,
    # overlapping amax and scale arrays; no groups is a no-op
    qg = lib.fp8_quantize_pertensor_grouped
    assert qg(one, -1, one, 8, 4, 4, one, 4, P(64), P(128), None) == -1
    assert qg(one, 1025, one, 8, 4, 4, one, 4, P(64), P(128), None) == -1
    assert qg(one, 2, None, 8, 4, 4, one, 4, P(64), P(128), None) == -1
    assert qg(one, 2, one, 8, 8, 4, one, 8, P(64), P(128), None) == -1
    assert qg(one, 4, one, 8, 4, 4, one, 4, P(64), P(72), None) == -1    # 16 B vs 8 B apart
    assert qg(one, 4, one, 8, 4, 4, one, 4, P(72), P(64), None) == -1
    assert qg(None, 0, None, 0, 4, 4, None, 4, None, None, None) == 0
    # timeout setter
    assert lib.fp8la_set_wait_timeout_ns(10) == -1
    assert lib.fp8la_set_wait_timeout_ns(2_000_000_000) == 0


def test_missing_library_fails_loudly():
    import precision_linear_algebra_gb300 as fl
    with pytest.raises(RuntimeError, match="not built"):
        fl.load(os.path.join(ROOT, "no_such_dir", "libfp8la.so"))


def test_no_cpu_fallback_without_a_gpu(lib):
    """Without a GPU every compute entry point returns an error before any
    launch and the binding raises; nothing is computed on the host."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: this checks the GPU-less behaviour")
    import precision_linear_algebra_gb300 as fl
    A = torch.zeros((32, 32), dtype=torch.uint8)
    B = torch.zeros((32, 32), dtype=torch.uint8)
    s = torch.ones(1)
    C = torch.full((32, 32), 7.0, dtype=torch.bfloat16)
    with pytest.raises(fl.Fp8laError) as e:
        fl.fp8_gemm(A.data_ptr(), 32, B.data_ptr(), 32, C.data_ptr(), 32, 32, 32, 32,
                    s.data_ptr(), s.data_ptr(), None)
    assert e.value.status in (-3, -4)
    assert torch.all(C == 7.0)
    x = torch.ones((4, 4))
    q = torch.zeros((4, 4), dtype=torch.uint8)
    s2 = torch.ones(1)
    with pytest.raises(fl.Fp8laError) as e:
        fl.fp8_quantize_pertensor(x.data_ptr(), 4, 4, 4, q.data_ptr(), 4, s.data_ptr(),
                                  s2.data_ptr(), None)
    assert e.value.status in (-3, -4)
    assert torch.all(q == 0)
