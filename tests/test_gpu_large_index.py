"""GPU parity past 2^31 elements: every kernel family on an input or output
whose flat element index exceeds the int32 range, checked against the oracle
on the rows, columns and blocks that lie past that point.

A kernel that formed any address with 32-bit arithmetic would write these
elements to the wrong place (or read the wrong input), which the sampled
comparisons below see as wrong bytes or a GEMM error far above the bar.

* Quantizers (blockwise 1x128 rowwise + colwise, MX 1x32 rowwise + colwise):
  x [524544, 4096] bf16, 2.149e9 elements; the last row block and columns
  (q[r, c] at r * 4096 + c, qT[c, r] at c * 524544 + r) and 128 random rows
  and columns elsewhere, byte for byte.
* Blockwise GEMMs: fwd and dgrad writing [262272, 8192] bf16 (2.149e9
  elements), wgrad writing dW [32768, 65792] in bf16 and in fp32 (2.156e9
  elements), on sampled rows and columns at the 2e-3 GEMM bar.
* MX grouped GEMM: FWD and DGRAD writing [262272, 8192] over two groups,
  WGRAD writing [2, 32768, 33024] (2.164e9 elements).

Inputs are seeded normals drawn on the device (x scaled per row by 2^U(-8, 8)
so the blocks' scales differ); only the sampled slices are copied to the host
for the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import f32, gemm_max_err, lib, u8
from mxfp8_precision_gemms_fp8bw_gb300 import binding as B

pytestmark = pytest.mark.gpu

TOL = oracle.GEMM_TOL
ACC_TOL = 1e-4
INT32_LIMIT = 2 ** 31


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()
    yield
    torch.cuda.empty_cache()


def _device_bf16(shape, seed, row_exp=8):
    """Seeded N(0, 1) bf16 on the device, rows scaled by exact powers of two."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device="cuda", dtype=torch.bfloat16)
    if row_exp:
        e = torch.randint(-row_exp, row_exp + 1, (shape[0], 1), generator=g, device="cuda")
        x.mul_(torch.exp2(e.float()).bfloat16())
    return x


def _idx(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).cuda()


def _tail_and_random(n: int, tail: int, extra: int, seed: int) -> np.ndarray:
    """The last `tail` indices of range(n) and `extra` distinct random ones before them, sorted."""
    rng = np.random.default_rng(seed)
    return np.sort(np.concatenate([np.arange(n - tail, n), rng.choice(n - tail, extra, replace=False)]))


# ---------------------------------------------------------------- quantizers

QR, QC = 524544, 4096          # 4098 x 32 blocks of 128; QR * QC > 2^31


@pytest.fixture(scope="module")
def big_x():
    assert QR * QC > INT32_LIMIT
    x = _device_bf16((QR, QC), seed=9001)
    yield x
    del x
    torch.cuda.empty_cache()


def test_blockwise_rowcol_quant_past_int32(big_x):
    x = big_x
    q = torch.empty((QR, QC), dtype=torch.uint8, device="cuda")
    s = torch.empty((QC // 128, QR), dtype=torch.float32, device="cuda")
    qT = torch.empty((QC, QR), dtype=torch.uint8, device="cuda")
    sT = torch.empty((QR // 128, QC), dtype=torch.float32, device="cuda")
    B.fp8bw_quant_1x128_rowcol(x, q, s, qT, sT)
    B.fp8bw_sync_status()

    rows = _tail_and_random(QR, 128, 128, seed=1)
    assert (rows[-1] * QC) > INT32_LIMIT
    ri = _idx(rows)
    q_ref, s_ref = oracle.quant_1x128_row(f32(x[ri]))
    assert np.array_equal(u8(q[ri]), q_ref)
    assert np.array_equal(f32(s[:, ri]).view(np.uint32), s_ref.view(np.uint32))

    cols = _tail_and_random(QC, 128, 128, seed=2)
    ci = _idx(cols)
    assert (cols[-1] * QR) > INT32_LIMIT
    for r0 in (QR - 128, 128 * 2048):
        qT_ref, sT_ref = oracle.quant_1x128_col(f32(x[r0:r0 + 128][:, ci]))
        assert np.array_equal(u8(qT[ci][:, r0:r0 + 128]), qT_ref)
        assert np.array_equal(f32(sT[r0 // 128][ci]).view(np.uint32), sT_ref[0].view(np.uint32))
    del q, s, qT, sT
    torch.cuda.empty_cache()


def test_mx_rowcol_quant_past_int32(big_x):
    x = big_x
    q = torch.empty((QR, QC), dtype=torch.uint8, device="cuda")
    e8 = torch.empty((QR, QC // 32), dtype=torch.uint8, device="cuda")
    qT = torch.empty((QC, QR), dtype=torch.uint8, device="cuda")
    e8T = torch.empty((QC, QR // 32), dtype=torch.uint8, device="cuda")
    B.mxfp8_quant_1x32_rowcol(x, q, e8, qT, e8T, B.MX_RCEIL)
    B.fp8bw_sync_status()

    rows = _tail_and_random(QR, 128, 128, seed=3)
    ri = _idx(rows)
    q_ref, e8_ref = oracle.mx_quant_1x32_row(f32(x[ri]), oracle.RCEIL)
    assert np.array_equal(u8(q[ri]), q_ref)
    assert np.array_equal(u8(e8[ri]), e8_ref)

    cols = _tail_and_random(QC, 128, 128, seed=4)
    ci = _idx(cols)
    for r0 in (QR - 128, 128 * 2048):
        qT_ref, e8T_ref = oracle.mx_quant_1x32_col(f32(x[r0:r0 + 128][:, ci]), oracle.RCEIL)
        assert np.array_equal(u8(qT[ci][:, r0:r0 + 128]), qT_ref)
        assert np.array_equal(u8(e8T[ci][:, r0 // 32:r0 // 32 + 4]), e8T_ref)
    del q, e8, qT, e8T
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- blockwise GEMMs

GM, GK, GN = 262272, 256, 8192   # fwd y [GM, GN] and dgrad dx [GM, GN]: > 2^31 elements


def _gpu_row_quant(t):
    q, s = B.alloc_quant_1x128_row(t)
    B.fp8bw_quant_1x128_row(t, q, s)
    return q, s


def _gpu_weight_quant(w):
    q, _, s = B.alloc_quant_128x128(w, False)
    B.fp8bw_quant_128x128(w, q, None, s)
    return q, s


def test_gemm_fwd_output_past_int32():
    assert GM * GN > INT32_LIMIT
    x = _device_bf16((GM, GK), seed=9101)
    w = _device_bf16((GN, GK), seed=9102, row_exp=0) * 0.02
    xq, xs = _gpu_row_quant(x)
    wq, ws = _gpu_weight_quant(w)
    y = torch.empty((GM, GN), dtype=torch.bfloat16, device="cuda")
    B.fp8bw_gemm_fwd(xq, xs, wq, ws, y)
    B.fp8bw_sync_status()

    rows = _tail_and_random(GM, 128, 128, seed=5)
    ri = _idx(rows)
    xq_o, xs_o = oracle.quant_1x128_row(f32(x[ri]))
    wq_o, _, ws_o = oracle.quant_128x128(f32(w))
    xd, wd = oracle.dequant_1x128_row(xq_o, xs_o), oracle.dequant_128x128(wq_o, ws_o)
    assert gemm_max_err(f32(y[ri]), xd @ wd.T, xd, wd) <= TOL
    del x, w, xq, xs, wq, ws, y
    torch.cuda.empty_cache()


def test_gemm_dgrad_output_past_int32():
    # dx [GM, GN] = dy [GM, GK] . W [GK, GN], W read from its stored codes.
    dy = _device_bf16((GM, GK), seed=9111)
    w = _device_bf16((GK, GN), seed=9112, row_exp=0) * 0.02
    dyq, dys = _gpu_row_quant(dy)
    wq, ws = _gpu_weight_quant(w)
    dx = torch.empty((GM, GN), dtype=torch.bfloat16, device="cuda")
    B.fp8bw_gemm_dgrad(dyq, dys, wq, None, ws, dx)
    B.fp8bw_sync_status()

    rows = _tail_and_random(GM, 128, 128, seed=6)
    ri = _idx(rows)
    dyq_o, dys_o = oracle.quant_1x128_row(f32(dy[ri]))
    wq_o, _, ws_o = oracle.quant_128x128(f32(w))
    a, wd = oracle.dequant_1x128_row(dyq_o, dys_o), oracle.dequant_128x128(wq_o, ws_o)
    assert gemm_max_err(f32(dx[ri]), a @ wd, a, wd.T) <= TOL
    del dy, w, dyq, dys, wq, ws, dx
    torch.cuda.empty_cache()


WM, WN, WK = 128, 32768, 65792   # dW [WN, WK]: > 2^31 elements, one contraction block


def test_gemm_wgrad_output_past_int32_bf16_and_fp32():
    assert WN * WK > INT32_LIMIT
    dy = _device_bf16((WM, WN), seed=9121) * 1e-3
    x = _device_bf16((WM, WK), seed=9122)
    dyqT, dysT = B.alloc_quant_1x128_col(dy)
    B.fp8bw_quant_1x128_col(dy, dyqT, dysT)
    xqT, xsT = B.alloc_quant_1x128_col(x)
    B.fp8bw_quant_1x128_col(x, xqT, xsT)
    dW = torch.empty((WN, WK), dtype=torch.bfloat16, device="cuda")
    B.fp8bw_gemm_wgrad(dyqT, dysT, xqT, xsT, dW)
    dW32 = torch.zeros((WN, WK), dtype=torch.float32, device="cuda")
    B.fp8bw_gemm_wgrad_acc_f32(dyqT, dysT, xqT, xsT, dW32)
    B.fp8bw_sync_status()

    ns = _tail_and_random(WN, 64, 64, seed=7)
    ks = _tail_and_random(WK, 128, 128, seed=8)
    assert ns[-1] * WK > INT32_LIMIT
    ni, ki = _idx(ns), _idx(ks)
    a_q = oracle.quant_1x128_col(f32(dy[:, ni]))
    b_q = oracle.quant_1x128_col(f32(x[:, ki]))
    a, b = oracle.dequant_1x128_row(*a_q), oracle.dequant_1x128_row(*b_q)
    ref = oracle.gemm_wgrad(*a_q, *b_q)
    got = dW[ni][:, ki]
    got32 = dW32[ni][:, ki]
    assert gemm_max_err(f32(got), ref, a, b) <= TOL
    assert gemm_max_err(f32(got32), ref, a, b, oracle.FP32_ROUNDOFF) <= ACC_TOL
    # From zero, the fp32 result rounded to bf16 is the bf16 wgrad output.
    assert torch.equal(got32.bfloat16(), got)
    del dy, x, dyqT, dysT, xqT, xsT, dW, dW32
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- MX grouped GEMM

def _mx_row(t):
    q, e8 = B.alloc_mx_row(t)
    B.mxfp8_quant_1x32_row(t, q, e8, B.MX_RCEIL)
    return q, e8


def test_mx_grouped_fwd_and_dgrad_output_past_int32():
    # Two groups of 131072 and 131200 tokens (multiples of 32).
    M, C, Nout, G = GM, GK, GN, 2
    group_end = np.array([131072, M], np.int32)
    ge = torch.from_numpy(group_end).cuda()
    x = _device_bf16((M, C), seed=9201)
    rows = _tail_and_random(M, 128, 0, seed=9)     # the last 128 rows: group 1
    rows0 = np.sort(np.random.default_rng(10).choice(int(group_end[0]), 128, replace=False))  # group 0
    xq, xe = _mx_row(x)

    # FWD: y [M, Nout] = x [M, C] . W_g^T, W [G, Nout, C] rowwise along C.
    w = _device_bf16((G * Nout, C), seed=9202, row_exp=0) * 0.02
    wq, we = _mx_row(w)
    y = torch.empty((M, Nout), dtype=torch.bfloat16, device="cuda")
    ws = B.alloc_grouped_workspace(0, G, M, Nout, C, "cuda")
    B.mxfp8_grouped_gemm(0, xq, xe, wq, we, ge, G, M, Nout, C, y, ws)
    B.fp8bw_sync_status()
    wf = f32(w).reshape(G, Nout, C)
    for g, r in ((1, rows), (0, rows0)):
        ri = _idx(r)
        a = oracle.mx_dequant_row(*oracle.mx_quant_1x32_row(f32(x[ri]), oracle.RCEIL))
        b = oracle.mx_dequant_row(*oracle.mx_quant_1x32_row(wf[g], oracle.RCEIL))
        assert gemm_max_err(f32(y[ri]), a @ b.T, a, b) <= TOL
    del y, ws, w, wq, we
    torch.cuda.empty_cache()

    # DGRAD: dx [M, Nout] = dy [M, C] . W_g with W [G, C, Nout], 3D colwise
    # (32-blocks along C) into W^T [G, Nout, C].
    dy = x
    w3 = _device_bf16((G * C, Nout), seed=9203, row_exp=0).reshape(G, C, Nout) * 0.02
    wqT, weT = B.alloc_mx_3d_col(w3)
    B.mxfp8_quant_3d_col(w3, wqT, weT, B.MX_RCEIL)
    dx = torch.empty((M, Nout), dtype=torch.bfloat16, device="cuda")
    ws = B.alloc_grouped_workspace(1, G, M, C, Nout, "cuda")
    B.mxfp8_grouped_gemm(1, xq, xe, wqT, weT, ge, G, M, C, Nout, dx, ws)
    B.fp8bw_sync_status()
    qT_o, e8T_o = oracle.mx_quant_3d_col(f32(w3), oracle.RCEIL)
    for g, r in ((1, rows), (0, rows0)):
        ri = _idx(r)
        a = oracle.mx_dequant_row(*oracle.mx_quant_1x32_row(f32(dy[ri]), oracle.RCEIL))
        b = oracle.mx_dequant_row(qT_o[g], e8T_o[g])      # [Nout, C]
        assert gemm_max_err(f32(dx[ri]), a @ b.T, a, b) <= TOL
    del x, xq, xe, w3, wqT, weT, dx, ws
    torch.cuda.empty_cache()


def test_mx_grouped_wgrad_output_past_int32():
    # dW [G, N, K] with G * N * K > 2^31; 256 tokens in two groups of 128.
    G, M, N, K = 2, 256, 32768, 33024
    assert G * N * K > INT32_LIMIT
    group_end = np.array([128, 256], np.int32)
    ge = torch.from_numpy(group_end).cuda()
    dy = _device_bf16((M, N), seed=9301) * 1e-3
    x = _device_bf16((M, K), seed=9302)
    dyqT, dyeT = B.alloc_mx_col(dy)
    B.mxfp8_quant_1x32_col(dy, dyqT, dyeT, B.MX_RCEIL)
    xqT, xeT = B.alloc_mx_col(x)
    B.mxfp8_quant_1x32_col(x, xqT, xeT, B.MX_RCEIL)
    dW = torch.empty((G, N, K), dtype=torch.bfloat16, device="cuda")
    ws = B.alloc_grouped_workspace(2, G, M, N, K, "cuda")
    B.mxfp8_grouped_gemm(2, dyqT, dyeT, xqT, xeT, ge, G, M, N, K, dW, ws)
    B.fp8bw_sync_status()

    ns = _tail_and_random(N, 64, 64, seed=11)
    ks = _tail_and_random(K, 128, 128, seed=12)
    ni, ki = _idx(ns), _idx(ks)
    a_all = oracle.mx_dequant_row(*oracle.mx_quant_1x32_col(f32(dy[:, ni]), oracle.RCEIL))   # [n, M]
    b_all = oracle.mx_dequant_row(*oracle.mx_quant_1x32_col(f32(x[:, ki]), oracle.RCEIL))    # [k, M]
    for g in range(G):
        lo, hi = (0, 128) if g == 0 else (128, 256)
        a, b = a_all[:, lo:hi], b_all[:, lo:hi]
        assert gemm_max_err(f32(dW[g][ni][:, ki]), a @ b.T, a, b) <= TOL
    del dy, x, dyqT, dyeT, xqT, xeT, dW, ws
    torch.cuda.empty_cache()
