"""GPU parity for the E5M2 variants: per-tensor quantisation to E5M2 (bit for
bit against the oracle) and GEMMs with E5M2 operands, alone or mixed with
E4M3 (within the same bound as the E4M3 GEMM)."""

import os

import numpy as np
import pytest

import _sweep
import oracle
from _helpers import bf16_to_f64, lib, to_dev
from precision_linear_algebra_gb300 import workloads

pytestmark = pytest.mark.gpu

FINITE = {"e4m3": np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8),
          "e5m2": np.array([c for c in range(256) if (c & 0x7C) != 0x7C], np.uint8)}


def _quantize(fl, x_np):
    import torch
    q, amax, scale = fl.quantize_pertensor(to_dev(x_np), fmt="e5m2")
    torch.cuda.synchronize()
    return q.cpu().numpy(), amax.item(), scale.item()


def _assert_same(x_np):
    fl = lib()
    q, amax, scale = _quantize(fl, x_np)
    rq, ramax, rscale = oracle.quantize_pertensor(x_np, fmt="e5m2")
    assert np.float32(amax).tobytes() == np.float32(ramax).tobytes()
    assert np.float32(scale).tobytes() == np.float32(rscale).tobytes()
    diff = np.flatnonzero(q.reshape(-1) != rq.reshape(-1))
    assert diff.size == 0, "codes differ at %d places, first: got %#x want %#x (x=%r)" % (
        diff.size, q.reshape(-1)[diff[0]], rq.reshape(-1)[diff[0]], x_np.reshape(-1)[diff[0]])


def test_quantize_e5m2_normal():
    A, _ = workloads.square(1024, seed=0)
    _assert_same(A)


def test_quantize_e5m2_specials():
    _assert_same(np.array([[0.0, -0.0, np.nan, 1e-30, -3.0, 2.0 ** -130, 57344.0, 7.0]],
                          dtype=np.float32))
    _assert_same(np.zeros((3, 5), np.float32))
    _assert_same(np.array([[np.inf, 2.0, -3.0, np.nan]], dtype=np.float32))


def _sweep_chunk(bits, vec4=True):
    """One chunk of fp32 bit patterns with 57344 appended (so that chunks
    within +-57344 run with qscale == 1 and test the cast alone); vec4 pads
    the row to a multiple of four values (the 16-byte path), else the scalar
    path runs."""
    tail = [57344.0, 0.0, 0.0, 0.0] if vec4 else [57344.0]
    x = np.concatenate([bits.view(np.float32), np.array(tail, np.float32)])[None, :]
    _assert_same(x)


def test_cast_sweep_e5m2_sampled():
    for top in (0x00, 0x37, 0x38, 0x46, 0x47, 0x80, 0xB8, 0xC7, 0x7F, 0xFF):
        lo = np.uint64(top) << np.uint64(24)
        bits = (np.arange(1 << 24, dtype=np.uint64) + lo).astype(np.uint32)
        _sweep_chunk(bits, vec4=True)
        _sweep_chunk(bits, vec4=False)


@pytest.mark.skipif(os.environ.get("FP8LA_QUICK") == "1",
                    reason="FP8LA_QUICK=1 leaves out the full 2^32 sweeps")
def test_cast_sweep_e5m2_exhaustive():
    """Every fp32 bit pattern through the 16-byte E5M2 quantiser path, bit
    for bit against the oracle (run in worker processes)."""
    fl = lib()
    _sweep.sweep_all("e5m2", lambda x: _quantize(fl, x))


@pytest.fixture(params=[1, 2, 4], ids=["single_cta", "cta_pair", "cta_quad"])
def variant(request):
    fl = lib()
    fl.fp8la_set_gemm_variant(request.param)
    yield request.param
    fl.fp8la_set_gemm_variant(0)


@pytest.mark.parametrize("fa,fb", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
@pytest.mark.parametrize("M,N,K", [(256, 512, 256), (300, 270, 208)])
def test_gemm_formats(fa, fb, M, N, K, variant):
    import torch
    fl = lib()
    rng = np.random.default_rng(M + N + K + len(fa + fb))
    A = rng.choice(FINITE[fa], size=(M, K)).astype(np.uint8)
    B = rng.choice(FINITE[fb], size=(N, K)).astype(np.uint8)
    sa, sb = np.float32(0.75), np.float32(0.003)
    C = fl.gemm(to_dev(A), to_dev(B), to_dev(np.array([sa])), to_dev(np.array([sb])),
                a_fmt=fa, b_fmt=fb)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    got = bf16_to_f64(C)
    r, Cref = oracle.gemm_pertensor(A, B, sa, sb, a_fmt=fa, b_fmt=fb)
    bound = oracle.tolerance_pertensor(A, B, sa, sb, r, a_fmt=fa, b_fmt=fb)
    assert np.all(np.isfinite(got))
    bad = np.abs(got - r) > bound
    assert not bad.any(), "%d outside the bound" % bad.sum()
    assert np.mean(got == oracle.bf16_bits_to_float(Cref)) > 0.99


def test_e5m2_end_to_end_quantize_gemm(variant):
    import torch
    fl = lib()
    A, B = workloads.square(512, seed=2)
    qa, _, sa = fl.quantize_pertensor(to_dev(A), fmt="e5m2")
    qb, _, sb = fl.quantize_pertensor(to_dev(B), fmt="e4m3")
    C = fl.gemm(qa, qb, sa, sb, a_fmt="e5m2", b_fmt="e4m3")
    torch.cuda.synchronize()
    rqa, _, rsa = oracle.quantize_pertensor(A, fmt="e5m2")
    rqb, _, rsb = oracle.quantize_pertensor(B)
    assert np.array_equal(qa.cpu().numpy(), rqa) and np.array_equal(qb.cpu().numpy(), rqb)
    r, _ = oracle.gemm_pertensor(rqa, rqb, rsa, rsb, a_fmt="e5m2", b_fmt="e4m3")
    bound = oracle.tolerance_pertensor(rqa, rqb, rsa, rsb, r, a_fmt="e5m2", b_fmt="e4m3")
    assert np.all(np.abs(bf16_to_f64(C) - r) <= bound)
