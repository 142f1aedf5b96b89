"""GPU parity of fp8bw_gemm_fwd_quant: y = x W^T with the 1x128 rowwise and
colwise quantizations of bf16(y) written by the GEMM's epilogue.

Everything is bit-exact: y equals fp8bw_gemm_fwd's output, and the codes and
fp32 scale bits equal the oracle's quantizers applied to that y (rowwise:
blocks of 128 columns of each row; colwise: blocks of 128 rows of each
column, written transposed).  Shapes run from one tile to more tiles than
SMs (so CTAs take several tiles and the epilogue's cross-warp handoff cycles
its barrier phases); x has all-zero rows and W all-zero rows, so y has
all-zero row and column blocks (scale EPS/448, codes 0).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import bits, f32, lib, u8
from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
from mxfp8_precision_gemms_fp8bw_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def _operands(M, K, N, seed):
    rng = np.random.default_rng(seed)
    x = inputs.normal_bf16(rng, (M, K), 1.0)
    w = inputs.normal_bf16(rng, (N, K), 0.02)
    x[rng.choice(M, max(1, M // 64), replace=False)] = 0          # zero rows of y
    w[rng.choice(N, max(1, N // 64), replace=False)] = 0          # zero columns of y
    xd, wd = x.cuda(), w.cuda()
    xq, xs = B.alloc_quant_1x128_row(xd)
    B.fp8bw_quant_1x128_row(xd, xq, xs)
    wq, wqT, ws = B.alloc_quant_128x128(wd, True)
    B.fp8bw_quant_128x128(wd, wq, wqT, ws)
    return xq, xs, wq, ws


@pytest.mark.parametrize("M,K,N,seed", [
    (128, 128, 256, 0),        # one tile
    (384, 640, 512, 1),        # several tiles, odd contraction-block count
    (2560, 256, 2048, 2),      # 160 tiles: more than SMs
    (4096, 2048, 8192, 3),     # the toy FFN's up-projection dims, ~7 tiles per CTA
])
def test_fwd_quant_bit_exact(M, K, N, seed):
    xq, xs, wq, ws = _operands(M, K, N, seed)
    dev = xq.device
    y_ref = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    B.fp8bw_gemm_fwd(xq, xs, wq, ws, y_ref)
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    yq, ys = B.alloc_quant_1x128_row(y)
    yqT, ysT = B.alloc_quant_1x128_col(y)
    B.fp8bw_gemm_fwd_quant(xq, xs, wq, ws, y, yq, ys, yqT, ysT)
    # rowwise-only form
    y1 = torch.empty_like(y)
    yq1, ys1 = B.alloc_quant_1x128_row(y)
    B.fp8bw_gemm_fwd_quant(xq, xs, wq, ws, y1, yq1, ys1)
    B.fp8bw_sync_status()
    assert torch.equal(y, y_ref) and torch.equal(y1, y_ref)
    yf = f32(y_ref)
    qo, so = oracle.quant_1x128_row(yf)
    assert np.array_equal(u8(yq), qo) and np.array_equal(bits(ys), bits(so))
    assert np.array_equal(u8(yq1), qo) and np.array_equal(bits(ys1), bits(so))
    qTo, sTo = oracle.quant_1x128_col(yf)
    assert np.array_equal(u8(yqT), qTo) and np.array_equal(bits(ysT), bits(sTo))
    # the zero blocks are there and came out as the rule says
    eps_scale = np.float32(np.float32(1e-12) / np.float32(448.0))
    assert np.any(so == eps_scale) and np.any(sTo == eps_scale)


def test_fwd_quant_feeds_the_next_linear():
    # y1 = x W1^T quantized in the epilogue feeds y2 = y1 W2^T: identical to
    # quantizing y1 with the stand-alone quantizer.
    M, K, H, N = 512, 256, 512, 256
    xq, xs, w1q, w1s = _operands(M, K, H, 4)
    rng = np.random.default_rng(5)
    w2 = inputs.normal_bf16(rng, (N, H), 0.02).cuda()
    w2q, _, w2s = B.alloc_quant_128x128(w2, False)
    B.fp8bw_quant_128x128(w2, w2q, None, w2s)
    y1 = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    q1, s1 = B.alloc_quant_1x128_row(y1)
    B.fp8bw_gemm_fwd_quant(xq, xs, w1q, w1s, y1, q1, s1)
    q1b, s1b = B.alloc_quant_1x128_row(y1)
    B.fp8bw_quant_1x128_row(y1, q1b, s1b)
    y2, y2b = (torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(2))
    B.fp8bw_gemm_fwd(q1, s1, w2q, w2s, y2)
    B.fp8bw_gemm_fwd(q1b, s1b, w2q, w2s, y2b)
    B.fp8bw_sync_status()
    assert torch.equal(q1, q1b) and torch.equal(s1, s1b) and torch.equal(y2, y2b)
