"""Test infrastructure: blockwise-scaled e4m3 quantizers and GEMMs of the CPU oracle.

Only tests, the package's ``smoke()`` entry and the bench's CPU-baseline leg
may import this module.  Nothing in the library path calls it.

What is computed (the Float8BlockwiseLinear training recipe):

* PR #2386 ("[not for land] float8 blockwise scaling training prototype using
  deep_gemm"), description: the forward and backward GEMMs of a dense linear
  on blockwise-scaled float8 operands; 128x128 scaling of the weight
  ("What I saw" and "path forward", item 2); the "128_1_128_128" GEMM used for
  forward/dgrad and the "128_1_128_1" GEMM used for grad_weight ("What I saw",
  torchtitan bullet).
* PR #4295 ("add FSDP and TP tests for Float8BlockwiseLinear"), review thread
  on the ``EPS = 1e-12`` constant and on ``BlockWise1x128`` scaling: 1x128
  blocks of activations and gradients along the contraction dimension, and the
  1e-12 floor on a block's largest magnitude.

Readings taken where the pages are silent (each also listed in the design
notes):

* scale rule: the block's largest magnitude, floored at EPS, is mapped onto
  e4m3's largest finite value: ``s = fl32(max(amax, EPS) / 448)``, and each
  element is stored as ``q = e4m3_rne_satfinite(fl32(x / s))`` -- an IEEE
  float32 division, not a multiply by a reciprocal;
* block names: forward and dgrad take the activation/gradient in 1x128 blocks
  along the contraction dim and the weight in 128x128 blocks; grad_weight
  takes both operands in 1x128 blocks along the token dim;
* dims must be multiples of 128 (no partial blocks);
* scale layouts: a 1x128 scale array is ``s[block][row]`` (contraction-block
  major); the 128x128 scale array is ``s[row_block][col_block]``, the layout
  PR #4295's ``_pad_blockwise_128x128_scale_k_major`` thread describes
  (K-major); its row stride padding is a layout detail the oracle omits.

Inputs are float32 arrays holding bf16 values (bf16 widens to float32 exactly).
GEMM results are float64 and unrounded; the library's bf16 outputs are compared
against them within the stated tolerance.
"""
from __future__ import annotations

import numpy as np

from .e4m3 import E4M3_MAX, e4m3_decode, e4m3_encode

# Floor on a block's largest magnitude (PR #4295, review thread on EPS).
EPS = np.float32(1e-12)
BLOCK = 128


def _check_f32(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype != np.float32:
        raise TypeError("oracle quantizers take float32 arrays holding bf16 values")
    return x


def block_scale(amax: np.ndarray) -> np.ndarray:
    """fp32 scale of a block from its largest magnitude: fl32(max(amax, EPS) / 448)."""
    amax = np.asarray(amax, dtype=np.float32)
    return (np.maximum(amax, EPS) / np.float32(E4M3_MAX)).astype(np.float32)


def quantize_with_scale(x: np.ndarray, s: np.ndarray) -> np.ndarray:
    """e4m3 codes of fl32(x / s) (broadcast s against x), IEEE float32 division."""
    v = (x / s).astype(np.float32)
    return e4m3_encode(v)


def quant_1x128_row(x: np.ndarray):
    """1x128 rowwise quantization of x[R, C] (BlockWise1x128 along the last dim).

    Returns ``q[R, C]`` (uint8 e4m3 codes) and ``s[C/128][R]`` (float32).
    """
    x = _check_f32(x)
    R, C = x.shape
    assert R % BLOCK == 0 and C % BLOCK == 0
    blocks = x.reshape(R, C // BLOCK, BLOCK)
    amax = np.abs(blocks).max(axis=2)                # [R, C/128], exact
    s = block_scale(amax)                            # [R, C/128]
    q = quantize_with_scale(blocks, s[:, :, None]).reshape(R, C)
    return q, np.ascontiguousarray(s.T)


def quant_1x128_col(x: np.ndarray):
    """1x128 colwise quantization of x[R, C]: blocks of 128 along R per column.

    This is the rowwise quantization of x transposed, and its outputs come in
    that transposed layout: ``qT[C, R]`` and ``s[R/128][C]``.  It feeds the
    grad_weight GEMM, whose contraction runs over the token dim (the
    "128_1_128_1" case of PR #2386).
    """
    x = _check_f32(x)
    return quant_1x128_row(np.ascontiguousarray(x.T))


def quant_128x128(x: np.ndarray):
    """128x128 block quantization of a weight W[R, C] (PR #2386, 128x128 scaling).

    Returns ``q[R, C]``, ``qT[C, R]`` (the same codes transposed) and
    ``s[R/128][C/128]``.
    """
    x = _check_f32(x)
    R, C = x.shape
    assert R % BLOCK == 0 and C % BLOCK == 0
    tiles = x.reshape(R // BLOCK, BLOCK, C // BLOCK, BLOCK)
    amax = np.abs(tiles).max(axis=(1, 3))            # [R/128, C/128]
    s = block_scale(amax)
    q = quantize_with_scale(tiles, s[:, None, :, None]).reshape(R, C)
    return q, np.ascontiguousarray(q.T), s


# --------------------------------------------------------------------------
# Dequantization and the three GEMMs.
# --------------------------------------------------------------------------

def dequant_1x128_row(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """float64 values of a rowwise-1x128 tensor: dec(q[r, c]) * s[c/128][r]."""
    R, C = q.shape
    return e4m3_decode(q) * np.repeat(s.astype(np.float64).T, BLOCK, axis=1)[:R, :C]


def dequant_128x128(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """float64 values of a 128x128-scaled tensor: dec(q[r, c]) * s[r/128][c/128]."""
    R, C = q.shape
    full = np.repeat(np.repeat(s.astype(np.float64), BLOCK, axis=0), BLOCK, axis=1)
    return e4m3_decode(q) * full[:R, :C]


def gemm_fwd(xq, xs, wq, ws) -> np.ndarray:
    """y[m, n] = sum_k x^[m, k] * W^[n, k] in float64 (y = x W^T).

    x^ = dequantized 1x128-rowwise x[M, K] (scales xs[K/128][M]); W^ =
    dequantized 128x128 W[N, K] (scales ws[N/128][K/128]).  Every product of
    an e4m3 value and an fp32 scale is exact in float64, so the only rounding
    is the float64 summation.
    """
    xd = dequant_1x128_row(xq, xs)
    wd = dequant_128x128(wq, ws)
    return xd @ wd.T


def gemm_dgrad(dyq, dys, wq, ws) -> np.ndarray:
    """dx[m, k] = sum_n dy^[m, n] * W^[n, k] in float64 (dx = dy W).

    dy^ = dequantized 1x128-rowwise dy[M, N] (scales dys[N/128][M]); W^ as in
    ``gemm_fwd``, now contracted over its row (N) index.
    """
    dyd = dequant_1x128_row(dyq, dys)
    wd = dequant_128x128(wq, ws)
    return dyd @ wd


def gemm_wgrad(dyqT, dysT, xqT, xsT) -> np.ndarray:
    """dW[n, k] = sum_m dy^[m, n] * x^[m, k] in float64 (dW = dy^T x).

    Both operands come from the colwise quantizer: dyqT[N, M] with scales
    dysT[M/128][N], and xqT[K, M] with scales xsT[M/128][K] -- 1x128 blocks
    along the token dim M on both sides (the "128_1_128_1" GEMM).
    """
    dyd = dequant_1x128_row(dyqT, dysT)              # [N, M]
    xd = dequant_1x128_row(xqT, xsT)                 # [K, M]
    return dyd @ xd.T
