"""Test infrastructure: the acceptance metrics the parity tests apply.

Only tests, the package's ``smoke()`` entry and the bench's CPU-baseline leg
may import this module.

* ``normalized_gemm_error``: for each output element, the error beyond the
  rounding of the exact result to the output format,
  max(|C_out[i, j] - C_ref[i, j]| - u * |C_ref[i, j]|, 0) / (||a^_i||_2 * ||b^_j||_2),
  where a^_i and b^_j are the dequantized contraction vectors of the two
  operands and u the output format's unit roundoff: 2^-8 for bf16 (8
  significant bits; e.g. C_ref = -67.7497 rounds to -67.5, an error of
  0.0037 |C|), 2^-24 for fp32.  Output rounding is a property of the output
  format, not of the blockwise accumulation, and by Cauchy-Schwarz
  (|C_ref| <= ||a^_i|| ||b^_j||) it alone could reach 2^-8 ~ 3.9e-3 of the
  normalizer on strongly correlated operands -- above the 2e-3 bar -- so it is
  allowed on top of that bar.  The tolerance the tests use is 2e-3.  Where the
  norm product is zero the reference is exactly zero and the output must be
  exactly zero too (reported as an infinite error otherwise).
* ``sqnr_db``: 10 log10(||ref||^2 / ||ref - out||^2), the end-to-end check of
  a quantized linear against the product of its unquantized bf16 inputs.
"""
from __future__ import annotations

import numpy as np

GEMM_TOL = 2e-3
SQNR_MIN_DB = 25.0
BF16_ROUNDOFF = 2.0 ** -8    # |bf16(c) - c| <= 2^-8 |c| for c in bf16's normal range
FP32_ROUNDOFF = 2.0 ** -24


def row_norms(a: np.ndarray) -> np.ndarray:
    """Euclidean norm of each row of a float64 matrix (the contraction vectors)."""
    a = np.asarray(a, dtype=np.float64)
    return np.sqrt(np.einsum("ij,ij->i", a, a))


def normalized_gemm_error(c_out, c_ref, a_norms, b_norms, out_roundoff: float = BF16_ROUNDOFF) -> np.ndarray:
    """Element-wise max(|c_out - c_ref| - out_roundoff * |c_ref|, 0) / (a_norms[:, None] * b_norms[None, :])."""
    c_out = np.asarray(c_out, dtype=np.float64)
    c_ref = np.asarray(c_ref, dtype=np.float64)
    denom = np.outer(np.asarray(a_norms, dtype=np.float64), np.asarray(b_norms, dtype=np.float64))
    diff = np.maximum(np.abs(c_out - c_ref) - out_roundoff * np.abs(c_ref), 0.0)
    with np.errstate(divide="ignore", invalid="ignore"):
        err = np.where(denom > 0, diff / np.where(denom > 0, denom, 1.0), np.where(diff == 0, 0.0, np.inf))
    return err


def sqnr_db(ref, out) -> float:
    ref = np.asarray(ref, dtype=np.float64)
    out = np.asarray(out, dtype=np.float64)
    sig = float(np.sum(ref * ref))
    noise = float(np.sum((ref - out) ** 2))
    if noise == 0.0:
        return float("inf")
    return 10.0 * np.log10(sig / noise)
