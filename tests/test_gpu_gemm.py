"""GPU parity of the three blockwise-scaled GEMMs against the float64 oracle.

Bar: max over elements of (|out - ref| - 2^-8 |ref|) / (||a_i|| ||b_j||) <=
2e-3 (the oracle's GEMM_TOL, with the bf16 output's own rounding, up to
2^-8 |ref|, allowed on top), and end-to-end SQNR >= 25 dB against the product
of the unquantized bf16 inputs.
Shapes span one tile, several tiles with more tiles than SMs, an odd number
of contraction blocks (wgrad over M = 384) with more tiles than SMs, the tiny
workload, and the full-size dense workload on sampled output rows.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import dense_inputs, f32, gemm_max_err, lib
from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
from mxfp8_precision_gemms_fp8bw_gb300 import inputs
from mxfp8_precision_gemms_fp8bw_gb300 import linear as L

pytestmark = pytest.mark.gpu

TOL = oracle.GEMM_TOL


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def gpu_linear(x, w, dy):
    xd, wd, dyd = x.cuda(), w.cuda(), dy.cuda()
    wq = L.quantize_weight(wd)
    y, _ = L.forward(xd, wq)
    dx, dW = L.backward(dyd, xd, wq)
    B.fp8bw_sync_status()
    return f32(y), f32(dx), f32(dW)


def oracle_linear(x, w, dy):
    xf, wf, dyf = f32(x), f32(w), f32(dy)
    xq, xs = oracle.quant_1x128_row(xf)
    wq, _, ws = oracle.quant_128x128(wf)
    dyq, dys = oracle.quant_1x128_row(dyf)
    dyqT, dysT = oracle.quant_1x128_col(dyf)
    xqT, xsT = oracle.quant_1x128_col(xf)
    y = oracle.gemm_fwd(xq, xs, wq, ws)
    dx = oracle.gemm_dgrad(dyq, dys, wq, ws)
    dW = oracle.gemm_wgrad(dyqT, dysT, xqT, xsT)
    deq = dict(x=oracle.dequant_1x128_row(xq, xs), w=oracle.dequant_128x128(wq, ws),
               dy=oracle.dequant_1x128_row(dyq, dys), dyT=oracle.dequant_1x128_row(dyqT, dysT),
               xT=oracle.dequant_1x128_row(xqT, xsT))
    return y, dx, dW, deq


def check_linear(x, w, dy, sqnr=True):
    y, dx, dW = gpu_linear(x, w, dy)
    yr, dxr, dWr, d = oracle_linear(x, w, dy)
    e_y = gemm_max_err(y, yr, d["x"], d["w"])
    e_dx = gemm_max_err(dx, dxr, d["dy"], d["w"].T)
    e_dW = gemm_max_err(dW, dWr, d["dyT"], d["xT"])
    assert e_y <= TOL and e_dx <= TOL and e_dW <= TOL, (e_y, e_dx, e_dW)
    if sqnr:
        xf, wf, dyf = (f32(t).astype(np.float64) for t in (x, w, dy))
        assert oracle.sqnr_db(xf @ wf.T, y) >= oracle.SQNR_MIN_DB
        assert oracle.sqnr_db(dyf @ wf, dx) >= oracle.SQNR_MIN_DB
        assert oracle.sqnr_db(dyf.T @ xf, dW) >= oracle.SQNR_MIN_DB
    return e_y, e_dx, e_dW


def test_tiny_linear_fwd_bwd():
    t = inputs.tiny()
    check_linear(t.x, t.w, t.dy)


@pytest.mark.parametrize("M,N,K,seed", [(128, 256, 256, 0), (384, 512, 768, 1), (256, 768, 1280, 2),
                                        (2048, 4096, 512, 3), (384, 4096, 1536, 4)])
def test_linear_shapes(M, N, K, seed):
    t = inputs.linear_inputs(M, K, N, seed=100 + seed)
    check_linear(t.x, t.w, t.dy)


def test_zero_inputs_give_exact_zero():
    M, N, K = 256, 256, 256
    z = torch.zeros((M, K), dtype=torch.bfloat16)
    w = inputs.linear_inputs(M, K, N, seed=7).w
    y, dx, dW = gpu_linear(z, w, torch.zeros((M, N), dtype=torch.bfloat16))
    assert np.all(y == 0) and np.all(dx == 0) and np.all(dW == 0)


def test_integer_operands_exact():
    # Codes of -1, 0, 1 with scales 1 or 2: every partial sum is an exact
    # integer in fp32 and every output an integer below 2^8 in magnitude, so
    # bf16 holds it exactly -- the GEMM must reproduce the oracle bit for bit.
    rng = np.random.default_rng(11)
    M, N, K = 256, 512, 384
    xq = oracle.e4m3_encode(rng.integers(-1, 2, size=(M, K)).astype(np.float32))
    wq = oracle.e4m3_encode(rng.integers(-1, 2, size=(N, K)).astype(np.float32))
    xs = np.exp2(rng.integers(0, 2, size=(K // 128, M))).astype(np.float32)
    ws = np.zeros((N // 128, B.scale_ld_128x128(K)), np.float32)
    ws[:, :K // 128] = np.exp2(rng.integers(0, 2, size=(N // 128, K // 128)))
    ref = oracle.gemm_fwd(xq, xs, wq, ws[:, :K // 128])
    assert np.all(np.abs(ref) < 256) and np.all(ref == np.round(ref))
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    B.fp8bw_gemm_fwd(torch.from_numpy(xq).cuda(), torch.from_numpy(xs).cuda(), torch.from_numpy(wq).cuda(),
                     torch.from_numpy(ws).cuda(), y)
    B.fp8bw_sync_status()
    assert np.array_equal(f32(y).astype(np.float64), ref)


# ---------------------------------------------------------------- full size (sampled)

def test_full_size_dense_sampled():
    t = dense_inputs()
    M, K = t.x.shape
    N = t.w.shape[0]
    y, dx, dW = gpu_linear(t.x, t.w, t.dy)
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(M, 128, replace=False))
    xf, wf, dyf = f32(t.x), f32(t.w), f32(t.dy)
    wq, _, ws = oracle.quant_128x128(wf)
    wdeq = oracle.dequant_128x128(wq, ws)
    xq, xs = oracle.quant_1x128_row(np.ascontiguousarray(xf[rows]))
    xdeq = oracle.dequant_1x128_row(xq, xs)
    assert gemm_max_err(y[rows], xdeq @ wdeq.T, xdeq, wdeq) <= TOL
    dyq, dys = oracle.quant_1x128_row(np.ascontiguousarray(dyf[rows]))
    dydeq = oracle.dequant_1x128_row(dyq, dys)
    assert gemm_max_err(dx[rows], dydeq @ wdeq, dydeq, wdeq.T) <= TOL
    # wgrad: 128 sampled rows n and 128 sampled columns k of dW (colwise
    # quantization is independent per column, so the oracle quantizes only those)
    ns = np.sort(rng.choice(N, 128, replace=False))
    ks = np.sort(rng.choice(K, 128, replace=False))
    dyT = oracle.quant_1x128_col(np.ascontiguousarray(dyf[:, ns]))
    xT = oracle.quant_1x128_col(np.ascontiguousarray(xf[:, ks]))
    a = oracle.dequant_1x128_row(*dyT)
    b = oracle.dequant_1x128_row(*xT)
    assert gemm_max_err(dW[np.ix_(ns, ks)], a @ b.T, a, b) <= TOL


def test_float8_blockwise_linear_module_autograd():
    # The nn.Linear replacement of PR #4295: forward and backward through autograd.
    t = inputs.tiny()
    layer = L.Float8BlockwiseLinear(512, 512, device="cuda")
    with torch.no_grad():
        layer.weight.copy_(t.w.cuda())
    x = t.x.cuda().requires_grad_(True)
    y = layer(x)
    y.backward(t.dy.cuda())
    torch.cuda.synchronize()
    yr, dxr, dWr, d = oracle_linear(t.x, t.w, t.dy)
    assert gemm_max_err(f32(y), yr, d["x"], d["w"]) <= TOL
    assert gemm_max_err(f32(x.grad), dxr, d["dy"], d["w"].T) <= TOL
    assert gemm_max_err(f32(layer.weight.grad), dWr, d["dyT"], d["xT"]) <= TOL


@pytest.mark.parametrize("M,N,K,seed", [(128, 128, 256, 0), (256, 384, 512, 1), (384, 1280, 2304, 2),
                                        (2048, 4096, 5120, 3)])
def test_dgrad_from_q_equals_dgrad_from_qT(M, N, K, seed):
    # dx = dy W computed from W's codes as stored ([N, K], read transposed by
    # the tensor core) and from the transposed copy ([K, N]): the same products
    # in the same order, so the same bits; and both within the bar of the oracle.
    t = inputs.linear_inputs(M, K, N, seed=400 + seed)
    dyd, wd = t.dy.cuda(), t.w.cuda()
    wq, wqT, ws = B.alloc_quant_128x128(wd, True)
    B.fp8bw_quant_128x128(wd, wq, wqT, ws)
    dyq, dys = B.alloc_quant_1x128_row(dyd)
    B.fp8bw_quant_1x128_row(dyd, dyq, dys)
    dx_q = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    dx_qT = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.fp8bw_gemm_dgrad(dyq, dys, wq, None, ws, dx_q)
    B.fp8bw_gemm_dgrad(dyq, dys, wq, wqT, ws, dx_qT)
    B.fp8bw_sync_status()
    assert torch.equal(dx_q, dx_qT)
    rows = np.arange(M) if M <= 512 else np.sort(np.random.default_rng(seed).choice(M, 256, replace=False))
    dyf, wf = f32(t.dy[rows]), f32(t.w)
    oq, os_ = oracle.quant_1x128_row(dyf)
    woq, _, wos = oracle.quant_128x128(wf)
    dd, wdq = oracle.dequant_1x128_row(oq, os_), oracle.dequant_128x128(woq, wos)
    assert gemm_max_err(f32(dx_q)[rows], dd @ wdq, dd, wdq.T) <= TOL


def _wgrad_case(M, N, K, seed):
    t = inputs.linear_inputs(M, K, N, seed=seed)
    dyd, xd = t.dy.cuda(), t.x.cuda()
    dyqT, dysT = B.alloc_quant_1x128_col(dyd)
    B.fp8bw_quant_1x128_col(dyd, dyqT, dysT)
    xqT, xsT = B.alloc_quant_1x128_col(xd)
    B.fp8bw_quant_1x128_col(xd, xqT, xsT)
    return t, dyqT, dysT, xqT, xsT


@pytest.mark.parametrize("M,N,K,seed", [(8192, 1536, 4096, 0), (5632, 1536, 4096, 1)])
def test_wgrad_split_tail(M, N, K, seed):
    # 192 output tiles: on 152 SMs the last 40 run as contraction parts (64 or
    # 44 blocks over 3 parts: lengths 21/21/22 and 14/15/15).  The parts' fp32
    # partials are added in part order, so two calls give the same bits; the
    # result is within the bar of the oracle.
    assert torch.cuda.get_device_properties(0).multi_processor_count == 152
    t, dyqT, dysT, xqT, xsT = _wgrad_case(M, N, K, 500 + seed)
    ws = B.alloc_wgrad_workspace(M, N, K, dyqT.device)
    assert ws is not None and ws.numel() > 0
    outs = []
    for _ in range(2):
        dW = torch.full((N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
        B.fp8bw_gemm_wgrad_ws(dyqT, dysT, xqT, xsT, dW, ws)
        B.fp8bw_sync_status()
        outs.append(dW)
    assert torch.equal(outs[0], outs[1])
    dq, ds = oracle.quant_1x128_col(f32(t.dy))
    xq, xs = oracle.quant_1x128_col(f32(t.x))
    dd, xdq = oracle.dequant_1x128_row(dq, ds), oracle.dequant_1x128_row(xq, xs)
    assert gemm_max_err(f32(outs[0]), dd @ xdq.T, dd, xdq) <= TOL
    # without a workspace the same call is the plain wgrad
    dW2 = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    B.fp8bw_gemm_wgrad_ws(dyqT, dysT, xqT, xsT, dW2, None)
    dW3 = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    B.fp8bw_gemm_wgrad(dyqT, dysT, xqT, xsT, dW3)
    B.fp8bw_sync_status()
    assert torch.equal(dW2, dW3)


def test_wgrad_split_large_token_against_whole_tiles():
    # The large-token wgrad (M = 128000 contracted, 240 output tiles: the last
    # 88 split in five contraction parts) against the whole-tile kernel on
    # every element.  (Its parity against the oracle is checked on sampled
    # outputs by the large-token linear test, which runs the same call.)
    M, K, N = 128000, 5120, 1536
    assert B.fp8bw_gemm_wgrad_workspace_bytes(M, N, K) > 0
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    dy = (torch.randn((M, N), generator=g, device="cuda") * 1e-3).bfloat16()
    x = torch.randn((M, K), generator=g, device="cuda").bfloat16()
    dyqT, dysT = B.alloc_quant_1x128_col(dy)
    B.fp8bw_quant_1x128_col(dy, dyqT, dysT)
    xqT, xsT = B.alloc_quant_1x128_col(x)
    B.fp8bw_quant_1x128_col(x, xqT, xsT)
    ws = B.alloc_wgrad_workspace(M, N, K, dy.device)
    dW = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    B.fp8bw_gemm_wgrad_ws(dyqT, dysT, xqT, xsT, dW, ws)
    # the tail's fp32 partial sums are added in another order (a difference of
    # a few fp32 ulps of the sum of |partials|, far below 1e-5 of the matrix's
    # largest value), which can move the bf16 rounding by one ulp (2^-7 of the
    # value); nothing else differs
    dW_plain = torch.empty_like(dW)
    B.fp8bw_gemm_wgrad(dyqT, dysT, xqT, xsT, dW_plain)
    B.fp8bw_sync_status()
    p = dW_plain.float()
    d = (dW.float() - p).abs()
    assert bool((d <= p.abs() * 2.0 ** -7 + 1e-5 * float(p.abs().max())).all())
    assert float((d > 0).float().mean()) < 0.01
