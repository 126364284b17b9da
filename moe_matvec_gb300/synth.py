"""Seeded synthetic inputs for the quantized matvec / MoE decode workloads.

This module only draws random numbers with the shapes and distributions of
the workloads; it holds none of the quantization or matvec arithmetic, so the
tests, the benchmark and the oracle can all consume the same inputs.

Workloads (decode-time shapes of the models the pages run, with
N(0, 0.02) weights and N(0, 1) activations):
  - q8_0_gemv   : Q8_0, M = K = 4096, 1 token
  - q4_k        : Q4_K, M = 17408, K = 5120, 1/2/4/8/16 tokens
  - iq4_xs      : IQ4_XS, 6144 x 2048 and 2048 x 6144, 1/4/8 tokens
  - moe         : 128 experts, top-8, hidden 4096, FFN 1536, gate/up IQ4_XS,
                  down Q4_K, 1/4/16/64 tokens; ids uniform without
                  replacement, gates = softmax of N(0,1) logits over the
                  chosen experts, renormalized
  - splitk_q8_0 : Q8_0, 151936 x 5120 (LM head) and 512 x 65536, 1..16 tokens
Seed recipe: 1000 * workload_index + 10 * shape_index + ntok_index; routing
draws use that seed + 7.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

WEIGHT_STD = 0.02


@dataclass(frozen=True)
class DenseCase:
    workload: str
    fmt: int
    M: int
    K: int
    n_toks: tuple
    index: int
    shape_index: int = 0


@dataclass(frozen=True)
class MoECase:
    workload: str = "moe"
    n_experts: int = 128
    top_k: int = 8
    hidden: int = 4096
    ffn: int = 1536
    fmt_gate_up: int = 2
    fmt_down: int = 1
    n_toks: tuple = (1, 4, 16, 64)
    index: int = 3


DENSE_CASES = (
    DenseCase("q8_0_gemv", 0, 4096, 4096, (1,), 0),
    DenseCase("q4_k", 1, 17408, 5120, (1, 2, 4, 8, 16), 1),
    DenseCase("iq4_xs", 2, 6144, 2048, (1, 4, 8), 2, 0),
    DenseCase("iq4_xs", 2, 2048, 6144, (1, 4, 8), 2, 1),
    DenseCase("splitk_q8_0", 0, 151936, 5120, (1, 2, 4, 8, 16), 4, 0),
    DenseCase("splitk_q8_0", 0, 512, 65536, (1, 2, 4, 8, 16), 4, 1),
)
MOE_CASE = MoECase()


def seed_for(index: int, shape_index: int, ntok_index: int) -> int:
    return 1000 * index + 10 * shape_index + ntok_index


def weights(seed: int, M: int, K: int, std: float = WEIGHT_STD) -> np.ndarray:
    """fp32 [M][K] ~ N(0, std^2)."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((M, K), dtype=np.float32)
    w *= np.float32(std)
    return w


def weight_rows(seed: int, M: int, K: int, rows, std: float = WEIGHT_STD) -> np.ndarray:
    """Rows `rows` of weights(seed, M, K) without drawing the whole matrix:
    each row comes from its own stream (seed, row), so any subset can be
    regenerated; this is a different matrix than weights(seed, M, K)."""
    out = np.empty((len(rows), K), np.float32)
    for i, r in enumerate(rows):
        rng = np.random.default_rng([seed, int(r)])
        out[i] = rng.standard_normal(K, dtype=np.float32) * np.float32(std)
    return out


def activations(seed: int, n: int, K: int) -> np.ndarray:
    """fp32 [n][K] ~ N(0, 1)."""
    rng = np.random.default_rng(seed + 1_000_003)
    return rng.standard_normal((n, K), dtype=np.float32)


def routing(seed: int, n: int, n_experts: int, top_k: int):
    """ids int32 [n][top_k] (a uniformly random ordered top_k-subset of the
    experts per token) and gates fp32 [n][top_k] (softmax of N(0,1) logits in
    fp64, rounded to fp32, then divided by their fp32 sum)."""
    rng = np.random.default_rng(seed + 7)
    ids = np.empty((n, top_k), np.int32)
    for t in range(n):
        ids[t] = rng.permutation(n_experts)[:top_k]
    logits = rng.standard_normal((n, top_k))
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    g = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    g = (g / g.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)
    return ids, g
