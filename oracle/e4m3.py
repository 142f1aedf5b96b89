"""Test infrastructure: the e4m3 codec of the CPU oracle.

Only tests, the package's ``smoke()`` entry and the bench's CPU-baseline leg
may import this module.  Nothing in the library path calls it.

The blockwise-FP8 recipe of PR #2386 ("[not for land] float8 blockwise scaling
training prototype using deep_gemm", description) and of PR #4295 ("add FSDP
and TP tests for Float8BlockwiseLinear", Summary) stores data as float8 e4m3.
The pages name the type only; its definition is the OCP 8-bit floating point
"E4M3" encoding:

* 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
* no infinities; S.1111.111 is NaN, so the largest finite magnitude is
  1.110b * 2^8 = 448 (code 0x7E);
* exponent field 0 holds subnormals k * 2^-9 (k = 0..7); the smallest normal
  is 2^-6 (code 0x08).

Rounding is round-to-nearest, ties to the even mantissa, of the real value of
the input, and a finite magnitude that rounds above 448 saturates to 448
("satfinite").  Every value is handled in float64, in which each float32 input
and each e4m3 value is exact, so no step of this codec rounds except the one
``np.rint`` that implements the e4m3 rounding itself.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0          # 1.110b * 2^8, code 0x7E
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_SUBNORMAL_QUANTUM = 2.0 ** -9


def e4m3_decode(codes) -> np.ndarray:
    """Value of each e4m3 code (uint8 array) as float64; NaN for S.1111.111."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp_field = (c >> 3) & 0xF
    mant = (c & 0x7).astype(np.float64)
    normal = sign * (1.0 + mant / 8.0) * np.ldexp(1.0, exp_field - 7)
    subnormal = sign * mant * E4M3_SUBNORMAL_QUANTUM
    out = np.where(exp_field == 0, subnormal, normal)
    out = np.where((c & 0x7F) == 0x7F, np.nan, out)
    return out


def e4m3_encode(v) -> np.ndarray:
    """e4m3 code of each value: round to nearest even, saturate finite to 448.

    ``v`` is a float32 (or float64) array.  NaN maps to 0x7F with the sign bit
    of the input; infinities saturate like any finite magnitude above 448
    (inputs of the quantizers are finite, so neither case is exercised by them).
    Signed zero is kept: -0.0 and negative values that round to zero give 0x80.
    """
    x = np.asarray(v, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)

    # Spacing of e4m3 values around a: 2^(floor(log2 a) - 3) in the normal
    # range, and the fixed subnormal spacing 2^-9 below 2^-6.  frexp gives the
    # exponent exactly: a = m * 2^ex with m in [0.5, 1), so floor(log2 a) = ex - 1.
    _, ex = np.frexp(a)
    e = np.maximum(ex - 1, -6)
    quantum = np.ldexp(1.0, e - 3)
    n = np.rint(a / quantum)            # a / quantum is exact; rint ties to even
    r = np.minimum(n * quantum, E4M3_MAX)   # saturate finite (and inf) to 448

    # Encode the rounded magnitude r, which is an e4m3 value.
    _, rex = np.frexp(r)
    r_exp = rex - 1                     # floor(log2 r) for r > 0
    is_normal = r >= E4M3_MIN_NORMAL
    safe_exp = np.where(is_normal, r_exp, 0)
    normal_code = ((safe_exp + 7) << 3) | (np.rint(r / np.ldexp(1.0, safe_exp) * 8.0) - 8.0).astype(np.int64)
    subnormal_code = np.rint(r / E4M3_SUBNORMAL_QUANTUM).astype(np.int64)
    code = np.where(is_normal, normal_code, subnormal_code)
    code = np.where(nan, 0x7F, code)
    code = code | np.where(neg, 0x80, 0)
    return code.astype(np.uint8)
