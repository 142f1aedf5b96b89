"""CPU oracle for the blockwise-FP8 / MXFP8 linear-layer training path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The library (``mxfp8_precision_gemms_fp8bw_gb300``) never imports it
and has no CPU fallback.

It is plain, slow numpy: every quantizer is the definition written out in
float32 (IEEE division, exact amax), the e4m3 codec is written from the OCP
format definition in float64, and every GEMM is one float64 matmul of the
dequantized operands.  It shares no code, table or constant generator with
the CUDA path.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, invariants, brute force on tiny inputs and independent
library codecs.  One quantity stays unpinned: the exact SQNR value reached on
the outlier-row FFN workload (only the 25 dB bound is checked).
"""
from .e4m3 import E4M3_MAX, e4m3_decode, e4m3_encode  # noqa: F401
from .blockwise import (  # noqa: F401
    EPS,
    block_scale,
    dequant_128x128,
    dequant_1x128_row,
    gemm_dgrad,
    gemm_fwd,
    gemm_wgrad,
    quant_128x128,
    quant_1x128_col,
    quant_1x128_row,
)
from .mx import (  # noqa: F401
    FLOOR,
    KIND_DGRAD,
    KIND_FWD,
    KIND_WGRAD,
    RCEIL,
    e8m0_exponent,
    group_starts,
    mx_dequant_row,
    mx_grouped_gemm,
    mx_quant_1x32_col,
    mx_quant_1x32_row,
    mx_quant_3d_col,
)
from .metrics import (BF16_ROUNDOFF, FP32_ROUNDOFF, GEMM_TOL, SQNR_MIN_DB, normalized_gemm_error,  # noqa: F401
                      row_norms, sqnr_db)
