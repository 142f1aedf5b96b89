"""Test infrastructure: MXFP8 quantizers and grouped GEMMs of the CPU oracle.

Only tests, the package's ``smoke()`` entry and the bench's CPU-baseline leg
may import this module.  Nothing in the library path calls it.

What is computed (PR #3037, "[mxfp8 moe training] use new 3d colwise
quantization kernel"):

* Summary: 3D expert weights are quantized colwise by a CUDA kernel whose
  output feeds the backward pass of the scaled grouped mm;
* Microbenchmarks table: grouped GEMMs of (M, N, K, G) with the
  ``MoEScalingType.MXFP8`` recipe, forward and forward+backward;
* review exchange at the end of the page: the colwise 3D quantization only
  affects the backward pass.

MXFP8 is taken in its plain meaning (the OCP Microscaling format): blocks of
32 consecutive elements along the contraction dim share one E8M0 scale (a
power of two 2^E stored as the byte E + 127), and each element is stored as
e4m3.  Readings taken where the pages are silent (also listed in the design
notes):

* exponent rule, mode RCEIL (0, default): E is the smallest integer with
  448 * 2^E >= amax -- the power-of-two counterpart of the blockwise rule
  "amax maps onto 448 without saturating"; mode FLOOR (1): the OCP MX rule
  E = floor(log2 amax) - 8 (8 being the exponent of e4m3's largest normal).
  E is clamped to [-127, 127]; an all-zero block gets E = -127 (byte 0x00);
* element rule: q = e4m3_rne_satfinite(fl32(x * 2^-E));
* "3D colwise" means blocks of 32 along dim 1 (N) of W[G, N, K] -- the dim the
  dgrad GEMM contracts -- stored per expert transposed: qT[G, K, N] with
  scales e8[G][K][N/32];
* the grouped GEMM's groups split the token dim M; group g owns tokens
  [group_end[g-1], group_end[g]) (group_end[-1] = 0); group sizes are
  multiples of 32 and may be zero.
"""
from __future__ import annotations

import numpy as np

from .e4m3 import E4M3_MAX, e4m3_decode, e4m3_encode

RCEIL = 0
FLOOR = 1
MX_BLOCK = 32
E8M0_BIAS = 127

KIND_FWD = 0
KIND_DGRAD = 1
KIND_WGRAD = 2


def e8m0_exponent(amax: np.ndarray, mode: int) -> np.ndarray:
    """Unbiased block exponent E (int64) from each block's largest magnitude."""
    a = np.asarray(amax, dtype=np.float64)          # float32 amax widens exactly
    pos = a > 0
    safe = np.where(pos, a, 1.0)
    if mode == RCEIL:
        # Smallest integer E with 448 * 2^E >= amax.  Start from a float
        # estimate and correct it with exact comparisons (448 * 2^E is exact
        # in float64 for the exponents that occur).
        E = np.floor(np.log2(safe / E4M3_MAX)).astype(np.int64)
        for _ in range(3):
            E = np.where(np.ldexp(E4M3_MAX, E - 1) >= safe, E - 1, E)
        for _ in range(3):
            E = np.where(np.ldexp(E4M3_MAX, E) < safe, E + 1, E)
    elif mode == FLOOR:
        # floor(log2 amax) - 8; frexp gives amax = m * 2^ex with m in [0.5, 1).
        _, ex = np.frexp(safe)
        E = ex.astype(np.int64) - 1 - 8
    else:
        raise ValueError("mode must be RCEIL (0) or FLOOR (1)")
    E = np.where(pos, E, -E8M0_BIAS)
    return np.clip(E, -E8M0_BIAS, E8M0_BIAS)


def mx_quant_1x32_row(x: np.ndarray, mode: int = RCEIL):
    """MXFP8 rowwise quantization of x[R, C] in 1x32 blocks along C.

    Returns ``q[R, C]`` (e4m3 codes) and ``e8[R][C/32]`` (biased E8M0 bytes).
    """
    x = np.asarray(x)
    if x.dtype != np.float32:
        raise TypeError("oracle quantizers take float32 arrays holding bf16 values")
    R, C = x.shape
    assert C % MX_BLOCK == 0
    blocks = x.reshape(R, C // MX_BLOCK, MX_BLOCK)
    amax = np.abs(blocks).max(axis=2)
    E = e8m0_exponent(amax, mode)                    # [R, C/32]
    scale_inv = np.ldexp(np.float32(1.0), (-E).astype(np.int32)).astype(np.float32)
    v = (blocks * scale_inv[:, :, None]).astype(np.float32)
    q = e4m3_encode(v).reshape(R, C)
    e8 = (E + E8M0_BIAS).astype(np.uint8)
    return q, e8


def mx_quant_1x32_col(x: np.ndarray, mode: int = RCEIL):
    """MXFP8 colwise quantization of x[R, C]: 32-blocks along R per column.

    The rowwise quantization of x transposed: ``qT[C, R]``, ``e8[C][R/32]``.
    """
    return mx_quant_1x32_row(np.ascontiguousarray(np.asarray(x).T), mode)


def mx_quant_3d_col(w: np.ndarray, mode: int = RCEIL):
    """3D colwise quantization of expert weights W[G, N, K] (32-blocks along N).

    Returns ``qT[G, K, N]`` and ``e8[G][K][N/32]``.
    """
    w = np.asarray(w)
    G = w.shape[0]
    outs = [mx_quant_1x32_col(w[g], mode) for g in range(G)]
    return np.stack([o[0] for o in outs]), np.stack([o[1] for o in outs])


def mx_dequant_row(q: np.ndarray, e8: np.ndarray) -> np.ndarray:
    """float64 values of a rowwise 1x32 tensor: dec(q[r, c]) * 2^(e8[r][c/32] - 127)."""
    E = e8.astype(np.int64) - E8M0_BIAS
    return e4m3_decode(q) * np.ldexp(1.0, np.repeat(E, MX_BLOCK, axis=-1))


def group_starts(group_end: np.ndarray) -> np.ndarray:
    ge = np.asarray(group_end, dtype=np.int64)
    return np.concatenate([[0], ge[:-1]])


def mx_grouped_gemm(kind: int, a, a_e8, b, b_e8, group_end, G: int, M: int, N: int, K: int) -> np.ndarray:
    """MoE grouped GEMM on MXFP8 operands, float64 result.

    The dims are those of the MoE linear: M tokens (split into G groups by
    ``group_end``), K input features, N output features per expert.

    * FWD   : a = x[M, K] rowwise, b = W[G, N, K] rowwise along K;
              y[m, n] = sum_k x^[m, k] W^_g[n, k] for m in group g  -> [M, N]
    * DGRAD : a = dy[M, N] rowwise, b = W^T[G, K, N] (3D colwise output);
              dx[m, k] = sum_n dy^[m, n] W^_g[n, k] for m in group g -> [M, K]
    * WGRAD : a = dy^T[N, M] colwise, b = x^T[K, M] colwise (32-blocks along M);
              dW_g[n, k] = sum_{m in group g} dy^[m, n] x^[m, k]  -> [G, N, K]
    """
    starts = group_starts(group_end)
    ends = np.asarray(group_end, dtype=np.int64)
    ad = mx_dequant_row(np.asarray(a), np.asarray(a_e8))
    bd = mx_dequant_row(np.asarray(b), np.asarray(b_e8))
    if kind == KIND_FWD or kind == KIND_DGRAD:
        n_out = N if kind == KIND_FWD else K
        bd = bd.reshape(G, n_out, -1)
        out = np.zeros((M, n_out), dtype=np.float64)
        for g in range(G):
            lo, hi = starts[g], ends[g]
            if hi > lo:
                out[lo:hi] = ad[lo:hi] @ bd[g].T
        return out
    if kind == KIND_WGRAD:
        out = np.zeros((G, N, K), dtype=np.float64)
        for g in range(G):
            lo, hi = starts[g], ends[g]
            if hi > lo:
                out[g] = ad[:, lo:hi] @ bd[:, lo:hi].T
        return out
    raise ValueError("kind must be FWD (0), DGRAD (1) or WGRAD (2)")
