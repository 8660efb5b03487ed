"""Seeded synthetic inputs for the FP8 quantize + GEMM workloads.

This module only draws random numbers (numpy PCG64 via default_rng); it does
none of the method's arithmetic, so the CPU oracle and the CUDA path can both
be fed from it.  Every draw happens in the order listed in each function.

Workloads (sizes as the method's evaluation fixes them):

* ``square(n, seed)``: A [n][n] ~ N(0,1), then B stored K-major [n][n]
  ~ N(0,1), fp32.  Used at n = 256 and n = 1024.
* ``square_outliers(n, seed)``: A ~ N(0,1), B ~ N(0, 0.02); then in each
  tensor 0.1% of entries (independent Bernoulli(0.001) per element) become
  exactly +-50 sigma (A: +-50.0, B: +-1.0) with a fair random sign.  Draw
  order: A base, B base, A mask, A signs, B mask, B signs.  Used at n = 8192.
* ``transformer_linear(name, seed)``: tokens M = 4096 (batch 2 x seq 2048)
  of a 70B-class decoder, hidden 8192, 64 heads x 128, 8 KV heads, FFN 28672:
  qkv (N 10240, K 8192), attn_out (8192, 8192), gate_up (57344, 8192),
  down (8192, 28672).  Activations [M][K] ~ N(0,1), weights [N][K] ~ N(0,0.02).
* ``moe_counts(seed)`` / ``moe_layer(seed)``: 8 experts, K 4096, N 14336,
  8192 tokens routed top-2 (16384 rows).  Per-expert row counts: expert
  probabilities p ~ Dirichlet(1, ..., 1), counts ~ Multinomial(16384, p); a
  count above 8192 (an expert cannot receive a token twice) is capped at 8192
  and the excess handed, one row at a time, to the expert with the fewest
  rows.  Activations [16384][4096] ~ N(0,1), grouped by expert in order;
  weights [8][14336][4096] ~ N(0,0.02).
"""

import numpy as np

TRANSFORMER_TOKENS = 4096
TRANSFORMER_LINEARS = {
    "qkv": (10240, 8192),
    "attn_out": (8192, 8192),
    "gate_up": (57344, 8192),
    "down": (8192, 28672),
}
MOE_EXPERTS = 8
MOE_K = 4096
MOE_N = 14336
MOE_TOKENS = 8192
MOE_TOPK = 2


def normal(rng, shape, sigma=1.0):
    x = rng.standard_normal(shape, dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    return x


def square(n, seed=0, m=None, k=None):
    """A [m][k] and B [n][k] (K-major), both N(0,1) fp32."""
    m = n if m is None else m
    k = n if k is None else k
    rng = np.random.default_rng(seed)
    A = normal(rng, (m, k))
    B = normal(rng, (n, k))
    return A, B


def _plant_outliers(rng, x, value):
    mask = rng.random(x.shape, dtype=np.float32) < np.float32(0.001)
    count = int(mask.sum())
    signs = rng.integers(0, 2, size=count).astype(np.float32) * 2 - 1
    x[mask] = signs * np.float32(value)
    return x


def square_outliers(n, seed=0):
    """A ~ N(0,1) and B ~ N(0,0.02), [n][n] each, with 0.1% +-50 sigma outliers."""
    rng = np.random.default_rng(seed)
    A = normal(rng, (n, n))
    B = normal(rng, (n, n), 0.02)
    A = _plant_outliers(rng, A, 50.0)
    B = _plant_outliers(rng, B, 50.0 * 0.02)
    return A, B


def transformer_linear(name, seed=0, tokens=TRANSFORMER_TOKENS):
    """Activations [tokens][K] ~ N(0,1), weights [N][K] ~ N(0,0.02)."""
    N, K = TRANSFORMER_LINEARS[name]
    rng = np.random.default_rng(seed)
    X = normal(rng, (tokens, K))
    W = normal(rng, (N, K), 0.02)
    return X, W


def moe_counts(seed=0, experts=MOE_EXPERTS, tokens=MOE_TOKENS, topk=MOE_TOPK):
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.ones(experts))
    counts = rng.multinomial(tokens * topk, p).astype(np.int64)
    excess = int(np.maximum(counts - tokens, 0).sum())
    counts = np.minimum(counts, tokens)
    while excess > 0:
        j = int(np.argmin(counts))
        counts[j] += 1
        excess -= 1
    return counts, rng


def moe_layer(seed=0, experts=MOE_EXPERTS, tokens=MOE_TOKENS, topk=MOE_TOPK,
              K=MOE_K, N=MOE_N):
    """(counts, m_offsets, activations [sum][K], weights [E][N][K])."""
    counts, rng = moe_counts(seed, experts, tokens, topk)
    m_offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    X = normal(rng, (int(m_offsets[-1]), K))
    W = normal(rng, (experts, N, K), 0.02)
    return counts, m_offsets, X, W
