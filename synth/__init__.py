"""Seeded synthetic inputs shared by the CPU oracle tests and the CUDA path.

This module draws random numbers and nothing else: it holds none of the
block-quantization arithmetic (no scale search, no packing, no decoding, no
dot products).  Both sides of every parity check take their inputs from here,
so the oracle and the GPU path see identical bytes.

Every generator uses numpy's PCG64 ``default_rng``.  Independent pieces of a
workload (weights, outlier columns, activations, routing ids, per-expert
weights) get their own child stream from ``SeedSequence(seed).spawn``, so a
test can draw one expert, or one small piece, without drawing the rest.

Workload shapes follow the LLM layers the source pages discuss: a decode FFN
projection (14336 x 4096), a 256-expert MoE bulk-expert matmul (768 x 2048 per
expert, top-8 routing), a prefill FFN matmul (17408 x 5120, 2048 tokens) and an
8192 x 8192 HFP4G32 matrix.  The pages' own models and evaluation suites are
not available; these seeded draws stand in for them.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "child_rngs",
    "normal_weights",
    "student_t_weights",
    "normal_activations",
    "outlier_bf16_activations",
    "routing_ids",
    "float32_to_bf16_bits",
    "bf16_bits_to_float32",
    "Workload",
    "tiny_gemv",
    "decode_gemv",
    "moe_gemv",
    "prefill_gemm",
    "hfp4_gemv",
]


def child_rngs(seed: int, n: int) -> list[np.random.Generator]:
    """``n`` independent PCG64 generators spawned from ``SeedSequence(seed)``."""
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


def normal_weights(rng: np.random.Generator, M: int, K: int, sigma: float) -> np.ndarray:
    """fp32 [M, K] with entries N(0, sigma^2)."""
    return (rng.standard_normal((M, K), dtype=np.float64) * sigma).astype(np.float32)


def student_t_weights(rng: np.random.Generator, M: int, K: int, nu: float = 5.0,
                      scale: float = 0.02) -> np.ndarray:
    """fp32 [M, K] with entries scale * t(nu) (heavy-tailed LLM-like weights)."""
    return (rng.standard_t(nu, size=(M, K)) * scale).astype(np.float32)


def outlier_columns(rng: np.random.Generator, K: int, frac: float = 0.01) -> np.ndarray:
    """round(frac*K) distinct column indices, drawn without replacement, sorted."""
    n = int(round(frac * K))
    return np.sort(rng.choice(K, size=n, replace=False)).astype(np.int64)


def normal_activations(rng: np.random.Generator, N: int, K: int) -> np.ndarray:
    """fp32 [N, K] with entries N(0, 1)."""
    return rng.standard_normal((N, K), dtype=np.float64).astype(np.float32)


def float32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); return uint16 bits.

    Inputs must be finite.  This is the input recipe's cast of the prefill
    activation matrix to bf16, not part of the quantized-weight method.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = ((u >> 16) & 1) + 0x7FFF
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_float32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bits to fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def outlier_bf16_activations(rng: np.random.Generator, N: int, K: int,
                             p: float = 0.005, mult: float = 20.0) -> np.ndarray:
    """bf16 bits [N, K]: N(0,1) entries, each scaled by ``mult`` with probability p."""
    x = rng.standard_normal((N, K), dtype=np.float64).astype(np.float32)
    mask = rng.random((N, K)) < p
    x[mask] *= np.float32(mult)
    return float32_to_bf16_bits(x)


def routing_ids(rng: np.random.Generator, T: int, top_k: int, E: int) -> np.ndarray:
    """int32 [T, top_k]: per token, top_k distinct experts drawn uniformly."""
    ids = np.empty((T, top_k), dtype=np.int32)
    for t in range(T):
        ids[t] = rng.choice(E, size=top_k, replace=False)
    return ids


class Workload(dict):
    """A dict of named numpy arrays plus a ``recipe`` string describing the draw."""

    def __init__(self, recipe: str, **arrays):
        super().__init__(**arrays)
        self.recipe = recipe


def tiny_gemv(M: int = 256, K: int = 1024, N: int = 1, seed: int = 0) -> Workload:
    """Small ROCmFP2 GEMV: W ~ N(0, 0.02^2) [M, K]; x ~ N(0, 1) [N, K]."""
    r_w, r_x = child_rngs(seed, 2)
    return Workload(
        f"W=N(0,0.02^2)[{M},{K}], x=N(0,1)[{N},{K}], seed={seed}",
        W=normal_weights(r_w, M, K, 0.02), x=normal_activations(r_x, N, K))


def decode_gemv(M: int = 14336, K: int = 4096, N: int = 1, seed: int = 1,
                outlier_frac: float = 0.01, outlier_mult: float = 8.0) -> Workload:
    """Decode FFN GEMV: W = 0.02 * t(5) [M, K] with round(1% K) columns x8; x ~ N(0,1).

    The activations are drawn as 8 rows and the first N are returned, so batch
    1 is the first row of batch 4.
    """
    r_w, r_c, r_x = child_rngs(seed, 3)
    W = student_t_weights(r_w, M, K)
    cols = outlier_columns(r_c, K, outlier_frac)
    W[:, cols] *= np.float32(outlier_mult)
    x = normal_activations(r_x, max(N, 8), K)[:N].copy()
    return Workload(
        f"W=0.02*t(5)[{M},{K}] with {len(cols)} columns x{outlier_mult:g}, "
        f"x=N(0,1)[{N},{K}], seed={seed}", W=W, x=x, outlier_cols=cols)


def moe_expert_weights(seed: int, E: int, M: int, K: int, e: int) -> np.ndarray:
    """Weights of expert ``e`` alone (its own child stream): 0.02 * t(5) [M, K]."""
    rng = np.random.default_rng(np.random.SeedSequence(seed).spawn(E + 2)[e])
    return student_t_weights(rng, M, K)


def moe_gemv(E: int = 256, M: int = 768, K: int = 2048, T: int = 16, top_k: int = 8,
             seed: int = 2, experts: bool = True) -> Workload:
    """MoE bulk-expert GEMV: E experts of 0.02*t(5) [M, K]; x ~ N(0,1) [T, K];
    ids [T, top_k] distinct per token, uniform.  ``experts=False`` skips the
    (large) weight draw; use :func:`moe_expert_weights` for single experts."""
    rngs = child_rngs(seed, E + 2)
    x = normal_activations(rngs[E], T, K)
    ids = routing_ids(rngs[E + 1], T, top_k, E)
    W = None
    if experts:
        W = np.empty((E, M, K), dtype=np.float32)
        for e in range(E):
            W[e] = student_t_weights(rngs[e], M, K)
    return Workload(
        f"E={E} experts of 0.02*t(5)[{M},{K}] (expert e from child stream e), "
        f"x=N(0,1)[{T},{K}], ids: {top_k} distinct of {E} per token, seed={seed}",
        W=W, x=x, ids=ids)


def prefill_gemm(M: int = 17408, K: int = 5120, N: int = 2048, seed: int = 3) -> Workload:
    """Prefill GEMM: W ~ N(0, 0.015^2) [M, K]; X bf16 [N, K] ~ N(0,1), 0.5% entries x20."""
    r_w, r_x = child_rngs(seed, 2)
    return Workload(
        f"W=N(0,0.015^2)[{M},{K}], X=bf16(N(0,1) with Bernoulli(0.005) x20)[{N},{K}], seed={seed}",
        W=normal_weights(r_w, M, K, 0.015), X=outlier_bf16_activations(r_x, N, K))


def hfp4_gemv(M: int = 8192, K: int = 8192, N: int = 1, seed: int = 4) -> Workload:
    """HFP4G32 GEMV: W ~ N(0, 0.02^2) [M, K]; x ~ N(0,1) drawn as 8 rows, first N used."""
    r_w, r_x = child_rngs(seed, 2)
    x = normal_activations(r_x, max(N, 8), K)[:N].copy()
    return Workload(f"W=N(0,0.02^2)[{M},{K}], x=N(0,1)[{N},{K}], seed={seed}",
                    W=normal_weights(r_w, M, K, 0.02), x=x)


def imatrix_importance(K: int, seed: int = 7, rows: int = 64) -> np.ndarray:
    """Synthetic importance per input column (an importance matrix stands in
    for calibration statistics): the mean of a^2 over `rows` activation rows
    whose channel scales are log-normal exp(N(0, 0.5^2)); fp32 [K]."""
    r_s, r_a = child_rngs(seed, 2)
    scale = np.exp(r_s.normal(0.0, 0.5, K))
    a = r_a.standard_normal((rows, K)) * scale
    return (a * a).mean(axis=0).astype(np.float32)
