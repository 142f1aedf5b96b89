"""Helpers of the GPU parity tests (not collected as tests)."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
from mxfp8_precision_gemms_fp8bw_gb300 import inputs


@functools.lru_cache(maxsize=1)
def dense_inputs():
    """The full-size dense linear workload, drawn once per test session."""
    return inputs.dense()


def lib():
    return B.lib(build_if_missing=True)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").float().numpy()


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").numpy()


def bits(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def adversarial_bf16(R: int, C: int, seed: int, block: int = 128) -> torch.Tensor:
    """bf16 [R, C] covering the quantizers' edge cases along rows of `block`s:
    per-row magnitudes across 2^+-60, all-zero and negative-zero blocks,
    constant blocks, bf16 subnormals, a lone huge outlier, blocks whose amax
    is 448*2^k holding exact e4m3 ties, and the division-vs-reciprocal case."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((R, C)).astype(np.float32)
    x *= np.exp2(rng.integers(-60, 61, size=(R, 1))).astype(np.float32)
    nb = C // block
    specials = [
        lambda b: np.zeros(block, np.float32),
        lambda b: np.full(block, -0.0, np.float32),
        lambda b: np.full(block, 3.25, np.float32),
        lambda b: (rng.standard_normal(block) * 1e-39).astype(np.float32),
        lambda b: np.concatenate([[1e30], rng.standard_normal(block - 1)]).astype(np.float32),
        lambda b: np.concatenate([[448.0 * 2.0 ** -3], rng.integers(-64, 65, size=block - 1) * 2.0 ** -5]).astype(np.float32),
        lambda b: np.concatenate([[392.0, 1.3671875, -1.3671875], rng.standard_normal(block - 3)]).astype(np.float32),
        lambda b: np.concatenate([[-448.0 * 4], (rng.integers(0, 16, size=block - 1) + 0.5) * 4]).astype(np.float32),
    ]
    for i, fn in enumerate(specials):
        r = (i * 37 + 5) % R
        b = (i * 3) % nb
        x[r, b * block:(b + 1) * block] = fn(b)
    return torch.from_numpy(x).to(torch.bfloat16)


def transpose_adversarial(R: int, C: int, seed: int, block: int = 128) -> torch.Tensor:
    """Same edge cases laid along columns (for the colwise quantizers)."""
    return adversarial_bf16(C, R, seed, block).t().contiguous()


def gemm_max_err(c_gpu: np.ndarray, c_ref: np.ndarray, a_deq: np.ndarray, b_deq: np.ndarray,
                 out_roundoff: float = oracle.BF16_ROUNDOFF) -> float:
    """Largest normalized error (see oracle.normalized_gemm_error) of an output
    whose format rounds with unit roundoff `out_roundoff` (bf16 unless given)."""
    err = oracle.normalized_gemm_error(c_gpu, c_ref, oracle.row_norms(a_deq), oracle.row_norms(b_deq), out_roundoff)
    return float(np.max(err))



def oracle_map(name: str, chunks, **kwargs):
    """oracle.<name>(*chunk, **kwargs) for every chunk, in a pool of spawned
    processes (safe after CUDA is initialised in this one; the workers import
    only numpy and the oracle); returns the results in order."""
    import concurrent.futures
    import multiprocessing
    import os

    import oracle_pool

    workers = max(1, min(len(chunks), (os.cpu_count() or 1)))
    ctx = multiprocessing.get_context("spawn")
    with concurrent.futures.ProcessPoolExecutor(max_workers=workers, mp_context=ctx) as ex:
        return list(ex.map(oracle_pool.call, [(name, c, kwargs) for c in chunks]))
