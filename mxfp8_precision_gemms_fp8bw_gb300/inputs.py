"""Seeded synthetic inputs for the blockwise-FP8 and MXFP8 linear workloads.

This module only draws random numbers and shapes them; it holds none of the
quantization or GEMM arithmetic, so both the CUDA path's tests/bench and the
CPU oracle's tests can take their inputs from it.

Random numbers come from numpy's PCG64 generator (``np.random.default_rng``),
whose float32 normal draws are reproducible across platforms; each draw is then
rounded to bf16 (round to nearest even) by torch.  "N(0, s)" means a normal
with standard deviation s.

Workloads (dims as in the MoE grouped-mm microbenchmark table of PR #3037 and
the ToyModel FFN of PR #4295):

* ``tiny``   -- x[256, 512] ~ N(0,1), W[512, 512] ~ N(0, 0.02),
                dy[256, 512] ~ N(0, 1e-3); seed 0; draw order x, W, dy.
* ``ffn``    -- tokens 4096, dim 2048, hidden 8192: x ~ N(0,1) with
                ceil(1%) = 41 rows multiplied by 10^U(1,2) (log-uniform in
                [10, 100]); w1, w2 [8192, 2048] and out_proj [2048, 8192] ~
                N(0, 0.02); dy[4096, 2048] ~ N(0, 1e-3); seed 1; draw order
                x, w1, w2, out_proj, dy, outlier rows (permutation), factors.
* ``dense``  -- M=16384, K=5120, N=8192, distributions as ``tiny``; seed 2.
* ``large``  -- M=128000 with (K, N) = (7168, 2048) or (5120, 1536); seed 3.
* ``moe``    -- M=16384 tokens over G=8 experts, K=5120, N=8192; group sizes
                32 * Multinomial(M/32, uniform over 8); x[M, K] ~ N(0,1),
                W[8, N, K] ~ N(0, 0.02), dy[M, N] ~ N(0, 1e-3); seed 4; draw
                order group sizes, x, W, dy.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

X_STD = 1.0
W_STD = 0.02
DY_STD = 1e-3


def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def normal_bf16(rng: np.random.Generator, shape, std: float) -> torch.Tensor:
    """A CPU bf16 tensor of N(0, std) draws (float32 draw, then RNE to bf16)."""
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return torch.from_numpy(a).to(torch.bfloat16)


@dataclass
class LinearInputs:
    x: torch.Tensor   # [M, K] bf16
    w: torch.Tensor   # [N, K] bf16
    dy: torch.Tensor  # [M, N] bf16


def linear_inputs(M: int, K: int, N: int, seed: int) -> LinearInputs:
    """x[M,K] ~ N(0,1), W[N,K] ~ N(0,0.02), dy[M,N] ~ N(0,1e-3), drawn in that order."""
    rng = _rng(seed)
    x = normal_bf16(rng, (M, K), X_STD)
    w = normal_bf16(rng, (N, K), W_STD)
    dy = normal_bf16(rng, (M, N), DY_STD)
    return LinearInputs(x, w, dy)


def tiny() -> LinearInputs:
    return linear_inputs(256, 512, 512, seed=0)


def dense() -> LinearInputs:
    return linear_inputs(16384, 5120, 8192, seed=2)


LARGE_SHAPES = ((128000, 7168, 2048), (128000, 5120, 1536))


def large(which: int = 0) -> LinearInputs:
    M, K, N = LARGE_SHAPES[which]
    return linear_inputs(M, K, N, seed=3)


@dataclass
class FFNInputs:
    x: torch.Tensor         # [4096, 2048]
    w1: torch.Tensor        # [8192, 2048]
    w2: torch.Tensor        # [8192, 2048]
    out_proj: torch.Tensor  # [2048, 8192]
    dy: torch.Tensor        # [4096, 2048]
    outlier_rows: np.ndarray
    outlier_factors: np.ndarray


def ffn(tokens: int = 4096, dim: int = 2048, hidden: int = 8192, seed: int = 1) -> FFNInputs:
    rng = _rng(seed)
    x = rng.standard_normal(size=(tokens, dim), dtype=np.float32)
    w1 = normal_bf16(rng, (hidden, dim), W_STD)
    w2 = normal_bf16(rng, (hidden, dim), W_STD)
    out_proj = normal_bf16(rng, (dim, hidden), W_STD)
    dy = normal_bf16(rng, (tokens, dim), DY_STD)
    n_out = -(-tokens // 100)                           # ceil(1% of rows)
    rows = rng.permutation(tokens)[:n_out]
    factors = np.power(10.0, rng.uniform(1.0, 2.0, size=n_out)).astype(np.float32)
    x[rows] *= factors[:, None]
    return FFNInputs(torch.from_numpy(x).to(torch.bfloat16), w1, w2, out_proj, dy, rows, factors)


@dataclass
class MoEInputs:
    group_end: np.ndarray   # int32 [G], cumulative token counts
    x: torch.Tensor         # [M, K]
    w: torch.Tensor         # [G, N, K]
    dy: torch.Tensor        # [M, N]


def moe_group_sizes(rng: np.random.Generator, M: int, G: int, align: int = 32) -> np.ndarray:
    counts = rng.multinomial(M // align, [1.0 / G] * G)
    return (counts * align).astype(np.int64)


def moe(M: int = 16384, K: int = 5120, N: int = 8192, G: int = 8, seed: int = 4) -> MoEInputs:
    rng = _rng(seed)
    sizes = moe_group_sizes(rng, M, G)
    x = normal_bf16(rng, (M, K), X_STD)
    w = normal_bf16(rng, (G, N, K), W_STD)
    dy = normal_bf16(rng, (M, N), DY_STD)
    return MoEInputs(np.cumsum(sizes).astype(np.int32), x, w, dy)


def bf16_to_f32_numpy(t: torch.Tensor) -> np.ndarray:
    """Exact float32 widening of a bf16 tensor, as a numpy array."""
    return t.detach().to("cpu").float().numpy()
