"""GPU parity of the MXFP8 grouped GEMM (FWD, DGRAD, WGRAD) against the oracle.

Bar: per output element |out - ref| / (||a_i|| ||b_j||) <= 2e-3 with a_i and
b_j the dequantized contraction vectors of that element's own group; empty
groups give exact zeros; invalid group tables are reported, never faulted on.
Group layouts cover boundaries that are multiples of 32 but not of 128, empty
groups first/middle/last, one group, and the full-size MoE workload (sampled).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import f32, lib, u8
from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
from mxfp8_precision_gemms_fp8bw_gb300 import inputs
from mxfp8_precision_gemms_fp8bw_gb300 import linear as L

pytestmark = pytest.mark.gpu
TOL = oracle.GEMM_TOL


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def gpu_moe(x, w, dy, group_end, mode=B.MX_RCEIL):
    xd, wd, dyd = x.cuda(), w.cuda(), dy.cuda()
    ge = torch.from_numpy(np.asarray(group_end, np.int32)).cuda()
    wq = L.mx_quantize_experts(wd, mode)
    y = L.mx_moe_forward(xd, wq, ge, mode)
    dx, dW = L.mx_moe_backward(dyd, xd, wq, ge, mode)
    B.fp8bw_sync_status()
    return f32(y), f32(dx), f32(dW)


def grouped_errors(x, w, dy, group_end, y, dx, dW, mode=B.MX_RCEIL, rows=None, n_sel=None, k_sel=None):
    """Max normalized error of y, dx, dW against the oracle, per group.

    rows / n_sel / k_sel restrict the check to sampled tokens, output features
    and input features; the oracle then quantizes only what those need (the
    rowwise and colwise MX blocks are independent per row / column)."""
    xf, wf, dyf = f32(x), f32(w), f32(dy)
    G, N, K = wf.shape
    n_sel = np.arange(N) if n_sel is None else np.asarray(n_sel)
    k_sel = np.arange(K) if k_sel is None else np.asarray(k_sel)
    starts = oracle.group_starts(group_end)
    e_y = e_dx = e_dW = 0.0
    sel = lambda a: np.ascontiguousarray(a)  # noqa: E731
    for g in range(G):
        lo, hi = int(starts[g]), int(group_end[g])
        if hi == lo:
            assert np.all(dW[g] == 0.0)
            continue
        r = np.arange(lo, hi) if rows is None else np.array([i for i in rows if lo <= i < hi], dtype=np.int64)
        if r.size:
            xd = oracle.mx_dequant_row(*oracle.mx_quant_1x32_row(sel(xf[r]), mode))
            wd = oracle.mx_dequant_row(*oracle.mx_quant_1x32_row(sel(wf[g][n_sel]), mode))       # [n, K]
            err = oracle.normalized_gemm_error(y[np.ix_(r, n_sel)], xd @ wd.T, oracle.row_norms(xd),
                                               oracle.row_norms(wd))
            e_y = max(e_y, float(err.max()))
            dyd = oracle.mx_dequant_row(*oracle.mx_quant_1x32_row(sel(dyf[r]), mode))
            wTd = oracle.mx_dequant_row(*oracle.mx_quant_1x32_col(sel(wf[g][:, k_sel]), mode))  # [k, N]
            err = oracle.normalized_gemm_error(dx[np.ix_(r, k_sel)], dyd @ wTd.T, oracle.row_norms(dyd),
                                               oracle.row_norms(wTd))
            e_dx = max(e_dx, float(err.max()))
        # wgrad of group g: colwise 1x32 of dy and x over the group's tokens
        a = oracle.mx_dequant_row(*oracle.mx_quant_1x32_col(sel(dyf[lo:hi][:, n_sel]), mode))
        b = oracle.mx_dequant_row(*oracle.mx_quant_1x32_col(sel(xf[lo:hi][:, k_sel]), mode))
        err = oracle.normalized_gemm_error(dW[g][np.ix_(n_sel, k_sel)], a @ b.T, oracle.row_norms(a),
                                           oracle.row_norms(b))
        e_dW = max(e_dW, float(err.max()))
    return e_y, e_dx, e_dW


def moe_inputs(M, K, N, group_end, seed):
    rng = np.random.default_rng(seed)
    G = len(group_end)
    x = inputs.normal_bf16(rng, (M, K), 1.0)
    w = inputs.normal_bf16(rng, (G, N, K), 0.02)
    dy = inputs.normal_bf16(rng, (M, N), 1e-3)
    return x, w, dy


@pytest.mark.parametrize("M,K,N,group_end", [
    (128, 256, 256, [128]),                         # one group, one tile
    (256, 256, 256, [96, 96, 256]),                 # empty middle group, 32-aligned boundary
    (384, 512, 512, [0, 160, 224, 384]),            # empty first group, short group
    (512, 256, 768, [32, 256, 512, 512]),           # 32-token group, empty last group
])
def test_grouped_small(M, K, N, group_end):
    x, w, dy = moe_inputs(M, K, N, group_end, seed=M + K)
    y, dx, dW = gpu_moe(x, w, dy, group_end)
    e = grouped_errors(x, w, dy, np.array(group_end), y, dx, dW)
    assert max(e) <= TOL, e


@pytest.mark.parametrize("seed", range(6))
def test_grouped_random_layouts(seed):
    # Seeded random expert counts, token splits (multiples of 32, empty groups
    # allowed) and dims; every group checked against the oracle.
    rng = np.random.default_rng(2000 + seed)
    G = int(rng.integers(1, 7))
    M = 32 * int(rng.integers(4, 65))
    K = 256 * int(rng.integers(1, 5))
    N = 256 * int(rng.integers(1, 5))
    sizes = 32 * rng.multinomial(M // 32, [1.0 / G] * G)
    ge = np.cumsum(sizes).astype(np.int32)
    x, w, dy = moe_inputs(M, K, N, ge, seed=3000 + seed)
    y, dx, dW = gpu_moe(x, w, dy, ge)
    e = grouped_errors(x, w, dy, ge, y, dx, dW)
    assert max(e) <= TOL, (G, M, K, N, list(sizes), e)


@pytest.mark.parametrize("N,group_end", [(384, [96, 96, 320]), (640, [128, 160, 512])])
def test_grouped_wgrad_odd_row_tiles(N, group_end):
    # WGRAD with N / 128 odd: dW's 128-row tiles cannot be paired, so the
    # unclustered kernel runs (every other shape pairs tiles that share B).
    M, K = int(group_end[-1]), 256
    G = len(group_end)
    rng = np.random.default_rng(N)
    x = inputs.normal_bf16(rng, (M, K), 1.0)
    dy = inputs.normal_bf16(rng, (M, N), 1e-3)
    xd, dyd = x.cuda(), dy.cuda()
    ge = torch.from_numpy(np.asarray(group_end, np.int32)).cuda()
    dyqT, dyeT = B.alloc_mx_col(dyd)
    B.mxfp8_quant_1x32_col(dyd, dyqT, dyeT)
    xqT, xeT = B.alloc_mx_col(xd)
    B.mxfp8_quant_1x32_col(xd, xqT, xeT)
    dW = torch.empty((G, N, K), dtype=torch.bfloat16, device="cuda")
    ws = B.alloc_grouped_workspace(B.GROUPED_WGRAD, G, M, N, K, xd.device)
    B.mxfp8_grouped_gemm(B.GROUPED_WGRAD, dyqT, dyeT, xqT, xeT, ge, G, M, N, K, dW, ws)
    B.fp8bw_sync_status()
    dWf, xf, dyf = f32(dW), f32(x), f32(dy)
    starts = oracle.group_starts(np.asarray(group_end))
    for g in range(G):
        lo, hi = int(starts[g]), int(group_end[g])
        if hi == lo:
            assert np.all(dWf[g] == 0.0)
            continue
        a = oracle.mx_dequant_row(*oracle.mx_quant_1x32_col(np.ascontiguousarray(dyf[lo:hi]), oracle.RCEIL))
        b = oracle.mx_dequant_row(*oracle.mx_quant_1x32_col(np.ascontiguousarray(xf[lo:hi]), oracle.RCEIL))
        err = oracle.normalized_gemm_error(dWf[g], a @ b.T, oracle.row_norms(a), oracle.row_norms(b))
        assert float(err.max()) <= TOL, (g, float(err.max()))


def test_grouped_floor_mode():
    M, K, N, ge = 256, 256, 256, [64, 256]
    x, w, dy = moe_inputs(M, K, N, ge, seed=5)
    y, dx, dW = gpu_moe(x, w, dy, ge, mode=B.MX_FLOOR)
    e = grouped_errors(x, w, dy, np.array(ge), y, dx, dW, mode=B.MX_FLOOR)
    assert max(e) <= TOL, e


def test_grouped_equals_dense_for_one_group_sqnr():
    M, K, N = 512, 512, 512
    x, w, dy = moe_inputs(M, K, N, [M], seed=9)
    y, dx, dW = gpu_moe(x, w, dy, [M])
    xf, wf, dyf = (f32(t).astype(np.float64) for t in (x, w, dy))
    assert oracle.sqnr_db(xf @ wf[0].T, y) >= oracle.SQNR_MIN_DB
    assert oracle.sqnr_db(dyf @ wf[0], dx) >= oracle.SQNR_MIN_DB
    assert oracle.sqnr_db(dyf.T @ xf, dW[0]) >= oracle.SQNR_MIN_DB


def test_invalid_group_table_is_reported():
    M, K, N = 256, 128, 256
    x, w, dy = moe_inputs(M, K, N, [100, 256], seed=3)
    xd, wd = x.cuda(), w.cuda()
    wq = L.mx_quantize_experts(wd)
    ge = torch.tensor([100, 256], dtype=torch.int32, device="cuda")   # 100 is not a multiple of 32
    y = L.mx_moe_forward(xd, wq, ge)
    with pytest.raises(B.Fp8bwError) as e:
        B.fp8bw_sync_status()
    assert e.value.code == B.ERR_SHAPE
    B.fp8bw_sync_status()   # cleared, context usable
    assert y.shape == (M, N)


def test_full_size_moe_sampled():
    t = inputs.moe()
    y, dx, dW = gpu_moe(t.x, t.w, t.dy, t.group_end)
    rng = np.random.default_rng(1)
    M, K = t.x.shape
    N = t.w.shape[1]
    rows = np.sort(rng.choice(M, 256, replace=False))
    n_sel = np.sort(rng.choice(N, 128, replace=False))
    k_sel = np.sort(rng.choice(K, 128, replace=False))
    e = grouped_errors(t.x, t.w, t.dy, t.group_end, y, dx, dW, rows=rows, n_sel=n_sel, k_sel=k_sel)
    assert max(e) <= TOL, e


def test_full_size_mxfp8_dense_linear_sampled():
    """The MXFP8 dense linear (the grouped path with one group, the mxfp8
    recipe of PR #3037's "Microbenchmarks" comparison) on the dense workload's
    x, W, dy (M=16384, K=5120, N=8192), checked on sampled rows and columns."""
    t = inputs.dense()
    M, K = t.x.shape
    N = t.w.shape[0]
    w3 = t.w.reshape(1, N, K)
    y, dx, dW = gpu_moe(t.x, w3, t.dy, [M])
    rng = np.random.default_rng(2)
    rows = np.sort(rng.choice(M, 256, replace=False))
    n_sel = np.sort(rng.choice(N, 128, replace=False))
    k_sel = np.sort(rng.choice(K, 128, replace=False))
    e = grouped_errors(t.x, w3, t.dy, np.array([M]), y, dx, dW, rows=rows, n_sel=n_sel, k_sel=k_sel)
    assert max(e) <= TOL, e
