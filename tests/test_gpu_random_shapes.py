"""Blockwise linear step on eight seeded random shapes (every dim a multiple of
128, output column counts multiples of 256; odd and even numbers of
contraction blocks, fewer and more tiles than SMs) against the oracle: the
quantized bytes bit-exact, each GEMM within the 2e-3 normalized bar."""
import numpy as np
import pytest

import oracle
from gpu_util import f32, gemm_max_err, lib
from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
from mxfp8_precision_gemms_fp8bw_gb300 import inputs
from mxfp8_precision_gemms_fp8bw_gb300 import linear as L

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def _shape(seed):
    rng = np.random.default_rng(1000 + seed)
    M = 128 * int(rng.integers(1, 33))     # 128 .. 4096 (1 .. 32 contraction blocks for wgrad)
    N = 256 * int(rng.integers(1, 17))     # 256 .. 4096
    K = 256 * int(rng.integers(1, 7))      # 256 .. 1536
    return M, N, K


@pytest.mark.parametrize("seed", range(8))
def test_random_shape_linear(seed):
    M, N, K = _shape(seed)
    t = inputs.linear_inputs(M, K, N, seed=500 + seed)
    x, w, dy = t.x.cuda(), t.w.cuda(), t.dy.cuda()
    ws = L.BlockwiseLinearWorkspace(M, N, K)
    y, dx, dW = ws.step(x, w, dy)
    B.fp8bw_sync_status()
    xf, wf, dyf = f32(t.x), f32(t.w), f32(t.dy)
    xq, xs = oracle.quant_1x128_row(xf)
    xqT, xsT = oracle.quant_1x128_col(xf)
    wq, wqT, wsc = oracle.quant_128x128(wf)
    dyq, dys = oracle.quant_1x128_row(dyf)
    dyqT, dysT = oracle.quant_1x128_col(dyf)
    assert np.array_equal(ws.xq.cpu().numpy(), xq) and np.array_equal(ws.xqT.cpu().numpy(), xqT)
    assert np.array_equal(ws.wq.cpu().numpy(), wq) and np.array_equal(ws.dyqT.cpu().numpy(), dyqT)
    xd, wd = oracle.dequant_1x128_row(xq, xs), oracle.dequant_128x128(wq, wsc)
    dyd = oracle.dequant_1x128_row(dyq, dys)
    a, b = oracle.dequant_1x128_row(dyqT, dysT), oracle.dequant_1x128_row(xqT, xsT)
    assert gemm_max_err(f32(y), oracle.gemm_fwd(xq, xs, wq, wsc), xd, wd) <= oracle.GEMM_TOL, (M, N, K)
    assert gemm_max_err(f32(dx), oracle.gemm_dgrad(dyq, dys, wq, wsc), dyd, wd.T) <= oracle.GEMM_TOL, (M, N, K)
    assert gemm_max_err(f32(dW), oracle.gemm_wgrad(dyqT, dysT, xqT, xsT), a, b) <= oracle.GEMM_TOL, (M, N, K)
