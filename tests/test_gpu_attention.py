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
        bound = oracle.bound_pertensor(r, K, sa[e], sb[e], np.abs(oracle.decode(A[rows])).max(),
                                       np.abs(oracle.decode(B[e])).max())
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
