"""GPU parity: the two GEMMs of FP8 multi-head attention (scores = Q K^T and
out = P V, per head, non-causal, head_dim 128) run as grouped GEMMs, one
group per head ([P2] "利用 Cutlass 内核命名惯例在 Triton 中实现 FP8 张量核的多头注意力
100 TFLOPS 加速", kernel paragraph: Q K^T with FP8 inputs and an FP32
accumulator; the softmax between the two GEMMs is not part of this path).

Layouts: Q [H*S][D] and K [H][S][D] are already K-major for Q K^T (the
contraction runs over D).  For P V the contraction runs over the key index,
so V enters transposed, [H][D][S]."""

import numpy as np
import pytest

import oracle
from _helpers import bf16_to_f64, lib, random_codes, to_dev

pytestmark = pytest.mark.gpu


def _grouped(fl, A, B, E, m_per, sa, sb):
    import torch
    offs = np.arange(E + 1, dtype=np.int32) * m_per
    C = fl.grouped_gemm(to_dev(offs), to_dev(A), to_dev(B), to_dev(sa), to_dev(sb))
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    return bf16_to_f64(C)


def _check(got, A, B, E, m_per, sa, sb):
    K = A.shape[1]
    for e in range(E):
        rows = slice(e * m_per, (e + 1) * m_per)
        r, Cref = oracle.gemm_pertensor(A[rows], B[e], sa[e], sb[e])
        bound = oracle.tolerance_pertensor(A[rows], B[e], sa[e], sb[e], r)
        assert np.all(np.abs(got[rows] - r) <= bound), "head %d" % e


@pytest.mark.parametrize("H,S", [(4, 256), (2, 384)])
def test_scores_and_pv_per_head(H, S):
    fl = lib()
    D = 128
    rng = np.random.default_rng(H * S)
    Q = random_codes(rng, (H * S, D))
    Kt = random_codes(rng, (H, S, D))
    sq = rng.uniform(0.01, 0.1, H).astype(np.float32)
    sk = rng.uniform(0.01, 0.1, H).astype(np.float32)
    scores = _grouped(fl, Q, Kt, H, S, sq, sk)            # [H*S][S]
    _check(scores, Q, Kt, H, S, sq, sk)
    P = random_codes(rng, (H * S, S))                     # quantised probabilities
    Vt = random_codes(rng, (H, D, S))                     # V transposed per head
    sp = rng.uniform(0.001, 0.01, H).astype(np.float32)
    sv = rng.uniform(0.01, 0.1, H).astype(np.float32)
    out = _grouped(fl, P, Vt, H, S, sp, sv)               # [H*S][D]
    _check(out, P, Vt, H, S, sp, sv)


def _codes_fast(rng, shape):
    """Uniform over the 254 finite E4M3 codes (all but 0x7F and 0xFF)."""
    x = rng.integers(0, 254, size=shape, dtype=np.uint8)
    return x + (x >= 0x7F).astype(np.uint8)


def test_full_size_sampled():
    """Batch 2 x 64 heads, sequence 2048, head_dim 128: both grouped GEMMs in
    the launch configuration of the attention benchmark (one group per head,
    128 groups of 2048 rows each), checked on sampled heads and rows against
    the oracle (every column of the sampled rows)."""
    import torch
    fl = lib()
    E, S, D = 128, 2048, 128
    rng = np.random.default_rng(2048)
    Q = _codes_fast(rng, (E * S, D))
    Kt = _codes_fast(rng, (E, S, D))
    P = _codes_fast(rng, (E * S, S))
    Vt = _codes_fast(rng, (E, D, S))
    sq, sk, sp, sv = (rng.uniform(0.001, 0.1, E).astype(np.float32) for _ in range(4))
    offs = to_dev(np.arange(E + 1, dtype=np.int32) * S)
    scores = fl.grouped_gemm(offs, to_dev(Q), to_dev(Kt), to_dev(sq), to_dev(sk))
    out = fl.grouped_gemm(offs, to_dev(P), to_dev(Vt), to_dev(sp), to_dev(sv))
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    for e in (0, 37, 90, 127):
        rows = np.sort(rng.choice(S, 24, replace=False))
        g = torch.from_numpy(e * S + rows).cuda()
        got_s = bf16_to_f64(scores.index_select(0, g))
        got_o = bf16_to_f64(out.index_select(0, g))
        A_s, A_o = Q[e * S:(e + 1) * S], P[e * S:(e + 1) * S]
        for got, A, B, sa, sb in ((got_s, A_s, Kt[e], sq[e], sk[e]),
                                  (got_o, A_o, Vt[e], sp[e], sv[e])):
            r, _ = oracle.gemm_pertensor(A, B, sa, sb, rows=rows)
            bound = oracle.tolerance_pertensor(A, B, sa, sb, r)
            assert np.all(np.isfinite(got)), "head %d" % e
            assert np.all(np.abs(got - r) <= bound), "head %d" % e
