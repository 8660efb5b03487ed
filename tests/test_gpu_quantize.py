"""GPU parity: quantisers against the oracle, bit for bit (codes and scales)."""

import os

import numpy as np
import pytest

import _sweep
import oracle
from _helpers import lib, to_dev
from precision_linear_algebra_gb300 import workloads

pytestmark = pytest.mark.gpu


def _run_pertensor(fl, x_np, ldx_pad=0, ldq_pad=0):
    import torch
    rows, cols = x_np.shape
    xs = torch.empty((rows, cols + ldx_pad), dtype=torch.float32, device="cuda")
    xs[:, :cols] = to_dev(x_np)
    qs = torch.full((rows, cols + ldq_pad), 0xA5, dtype=torch.uint8, device="cuda")
    x = xs[:, :cols]
    q = qs[:, :cols]
    q_out, amax, scale = fl.quantize_pertensor(x, q=q)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    if ldq_pad:
        assert torch.all(qs[:, cols:] == 0xA5), "write outside the row"
    return q.cpu().numpy(), amax.item(), scale.item()


def _assert_same(got, x_np):
    q, amax, scale = got
    rq, ramax, rscale = oracle.quantize_pertensor(x_np)
    assert np.float32(amax).tobytes() == np.float32(ramax).tobytes()
    assert np.float32(scale).tobytes() == np.float32(rscale).tobytes()
    diff = np.flatnonzero(q.reshape(-1) != rq.reshape(-1))
    assert diff.size == 0, "codes differ at %d places, first %d: got %#x want %#x (x=%r)" % (
        diff.size, diff[0], q.reshape(-1)[diff[0]], rq.reshape(-1)[diff[0]], x_np.reshape(-1)[diff[0]])


@pytest.mark.parametrize("n", [256, 1024])
def test_pertensor_square_configs(n):
    fl = lib()
    A, B = workloads.square(n, seed=0)
    for x in (A, B):
        _assert_same(_run_pertensor(fl, x), x)


@pytest.mark.parametrize("shape,ldx_pad,ldq_pad", [
    ((1, 1), 0, 0), ((1, 3), 0, 0), ((7, 13), 0, 0), ((33, 64), 0, 0),
    ((65, 100), 4, 16), ((3, 17), 3, 5), ((1000, 1001), 0, 0), ((5, 4096), 0, 0)])
def test_pertensor_ragged_and_strided(shape, ldx_pad, ldq_pad):
    fl = lib()
    rng = np.random.default_rng(hash(shape) & 0xFFFF)
    x = (rng.standard_normal(shape) * 3).astype(np.float32)
    _assert_same(_run_pertensor(fl, x, ldx_pad, ldq_pad), x)


@pytest.mark.parametrize("shape", [(1, 4), (3, 4096), (512, 1024), (513, 1024), (1024, 1028)])
def test_pertensor_one_launch_path_threshold(shape):
    """Contiguous tensors of up to 512K floats take the one-launch cluster
    path (no memset, amax exchanged through distributed shared memory);
    larger ones the two-pass grid path.  Both sides of the size limit."""
    fl = lib()
    rng = np.random.default_rng(shape[0] * 31 + shape[1])
    x = (rng.standard_normal(shape) * 7).astype(np.float32)
    x.reshape(-1)[rng.integers(0, x.size)] = -1234.5     # the amax, negative
    _assert_same(_run_pertensor(fl, x), x)


def test_pertensor_special_values():
    fl = lib()
    x = np.array([[0.0, -0.0, np.nan, 1e-30, -1e-30, 3.0, -7.0, 2.0 ** -130, 448.0, -5.5]],
                 dtype=np.float32)
    _assert_same(_run_pertensor(fl, x), x)
    z = np.zeros((4, 8), dtype=np.float32)
    _assert_same(_run_pertensor(fl, z), z)
    tiny = np.array([[1e-39, -5e-40, 0.0, 3e-45]], dtype=np.float32)
    _assert_same(_run_pertensor(fl, tiny), tiny)
    inf = np.array([[np.inf, 2.0, -3.0, np.nan]], dtype=np.float32)
    _assert_same(_run_pertensor(fl, inf), inf)


def test_pertensor_empty_writes_unit_scale():
    import torch
    fl = lib()
    x = torch.empty((0, 16), dtype=torch.float32, device="cuda")
    q, amax, scale = fl.quantize_pertensor(x)
    torch.cuda.synchronize()
    assert amax.item() == 0.0 and scale.item() == 1.0


def test_pertensor_8192_outliers_full_size():
    """The 8192^2 operands with 0.1% +-50 sigma outliers, bit for bit."""
    fl = lib()
    A, B = workloads.square_outliers(8192, seed=0)
    for x in (A, B):
        _assert_same(_run_pertensor(fl, x), x)


def _sweep_chunk(fl, bits, vec4=True):
    """Quantise one chunk of fp32 bit patterns with 448 appended (so that
    chunks whose patterns stay within +-448 run with qscale == 1 and test the
    cast alone) and compare with the oracle.  vec4: pad the row to a multiple
    of four values so that the 16-byte path (the one every aligned tensor
    takes, with its paired conversions) runs; otherwise the scalar path."""
    tail = [448.0, 0.0, 0.0, 0.0] if vec4 else [448.0]
    x = np.concatenate([bits.view(np.float32), np.array(tail, np.float32)])[None, :]
    _assert_same(_run_pertensor(fl, x), x)


def test_cast_sweep_sampled():
    """All fp32 patterns of selected exponent ranges (subnormals, the E4M3
    subnormal/normal boundary, the saturation range) plus a random sample."""
    fl = lib()
    for top in (0x00, 0x3A, 0x3B, 0x3C, 0x3D, 0x43, 0x80, 0xBB, 0xC3, 0x7F, 0xFF):
        lo = np.uint64(top) << np.uint64(24)
        bits = (np.arange(1 << 24, dtype=np.uint64) + lo).astype(np.uint32)
        _sweep_chunk(fl, bits, vec4=True)
        _sweep_chunk(fl, bits, vec4=False)
    rng = np.random.default_rng(99)
    _sweep_chunk(fl, rng.integers(0, 2 ** 32, size=1 << 24, dtype=np.uint64).astype(np.uint32))


@pytest.mark.skipif(os.environ.get("FP8LA_QUICK") == "1",
                    reason="FP8LA_QUICK=1 leaves out the full 2^32 sweeps")
def test_cast_sweep_exhaustive():
    """Every fp32 bit pattern through the 16-byte quantiser path, 2^24 at a
    time, bit for bit against the oracle (run in worker processes)."""
    fl = lib()
    _sweep.sweep_all("e4m3", lambda x: _run_pertensor(fl, x))


@pytest.mark.parametrize("shape,pad", [((64, 64), 0), ((70, 100), 0), ((33, 31), 5),
                                       ((96, 4096), 8), ((1, 1), 0), ((257, 129), 3)])
def test_blockwise_32x32(shape, pad):
    import torch
    fl = lib()
    rng = np.random.default_rng(shape[0] * 1000 + shape[1])
    x = (rng.standard_normal(shape) * rng.choice([0.01, 1, 100], size=shape)).astype(np.float32)
    x[0, 0] = 77.0
    rows, cols = shape
    xs = torch.zeros((rows, cols + pad), dtype=torch.float32, device="cuda")
    xs[:, :cols] = to_dev(x)
    q, s = fl.quantize_blockwise_32x32(xs[:, :cols])
    torch.cuda.synchronize()
    rq, rs = oracle.quantize_blockwise_32x32(x)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def test_blockwise_transformer_weights_sampled():
    """gate_up weights [57344][8192] ~ N(0,0.02): full GPU pass, oracle on
    sampled 32-aligned tile regions."""
    import torch
    fl = lib()
    X, W = workloads.transformer_linear("gate_up", seed=0, tokens=64)
    q, s = fl.quantize_blockwise_32x32(to_dev(W))
    torch.cuda.synchronize()
    qn, sn = q.cpu().numpy(), s.cpu().numpy()
    rng = np.random.default_rng(5)
    for _ in range(8):
        r0 = int(rng.integers(0, W.shape[0] // 32 - 2)) * 32
        c0 = int(rng.integers(0, W.shape[1] // 32 - 2)) * 32
        rq, rs = oracle.quantize_blockwise_32x32(W[r0:r0 + 64, c0:c0 + 64])
        assert np.array_equal(qn[r0:r0 + 64, c0:c0 + 64], rq)
        assert np.array_equal(sn[r0 // 32:r0 // 32 + 2, c0 // 32:c0 // 32 + 2], rs)


def _special_tiles():
    """A [101][136] fp32 array whose 32 x 32 tiles hold the degenerate cases
    of the per-tile scale rule: all zeros, signed zeros, +Inf and -Inf (amax
    Inf: qscale 0, scale Inf), NaN (ignored by the amax, coded 0x7F), fp32
    subnormals only (448/amax overflows: qscale = scale = 1), values near the
    fp32 maximum, values that land exactly on 448 and on E4M3 rounding
    midpoints; the last tile row and column are ragged."""
    rng = np.random.default_rng(77)
    x = (rng.standard_normal((101, 136)) * 3).astype(np.float32)
    t = lambda i, j: (slice(32 * i, 32 * i + 32), slice(32 * j, 32 * j + 32))
    x[t(0, 0)] = 0.0
    x[t(0, 1)] = -0.0
    x[t(0, 1)][5, 7] = 0.0
    x[t(0, 2)][3, 3] = np.inf
    x[t(0, 3)][31, 0] = -np.inf
    x[t(0, 3)][0, 31] = np.nan
    x[t(1, 0)][:, :] = np.nan
    x[t(1, 0)][4, 4] = 2.5
    x[t(1, 1)] = rng.standard_normal((32, 32)).astype(np.float32) * np.float32(1e-40)
    x[t(1, 2)] = (rng.uniform(-3.0, 3.0, (32, 32)) * 1e38).astype(np.float32)
    x[t(1, 2)][0, 0] = np.float32(3.4e38)
    # amax 448: the codes are the values themselves, including midpoints
    # between E4M3 neighbours (ties to even)
    mids = np.array([448.0, -448.0, 1.0625, 1.1875, 17.0, 19.0, 0.001953125 * 1.5,
                     240.0, 232.0, 0.5], np.float32)
    x[t(1, 3)] = 0.25
    x[t(1, 3)][0, :mids.size] = mids
    x[t(2, 4)][0, 0] = np.inf            # ragged corner tile (rows 96..100, cols 128..135)
    return x


def test_blockwise_special_tiles():
    import torch
    fl = lib()
    x = _special_tiles()
    xs = torch.zeros((x.shape[0], x.shape[1] + 4), dtype=torch.float32, device="cuda")
    xs[:, :x.shape[1]] = to_dev(x)
    for view in (xs[:, :x.shape[1]], to_dev(x)):      # padded stride, then contiguous
        q, s = fl.quantize_blockwise_32x32(view)
        torch.cuda.synchronize()
        assert fl.device_status() == 0
        rq, rs = oracle.quantize_blockwise_32x32(x)
        got_q = q.cpu().numpy()
        diff = np.argwhere(got_q != rq)
        assert diff.size == 0, "codes differ at %d places, first %s: got %#x want %#x" % (
            len(diff), tuple(diff[0]), got_q[tuple(diff[0])], rq[tuple(diff[0])])
        assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    # the cases the array is meant to hold
    assert rs[0, 0] == 1.0 and rs[0, 2] == np.inf and rs[1, 1] == 1.0 and rs[1, 3] == 1.0
    assert np.isfinite(rs[1, 2]) and rs[2, 4] == np.inf
    assert np.all(rq[32:64, 0:32][np.isnan(x[32:64, 0:32])] == 0x7F)
