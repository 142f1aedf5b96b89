"""The toy FFN workload (PR #4295's ToyModel: w1, w2 up-projections and
out_proj, tokens 4096, dim 2048, hidden 8192, 1 % outlier rows in x) forward
and backward through Float8BlockwiseLinear GEMMs, and the large-token dense
workloads (M = 128000) whose wgrad contracts over 128000 tokens.

* GEMMs fed directly by the workload's inputs are checked against the oracle
  element by element (normalized error <= 2e-3).
* The whole FFN step is run a second time through the oracle (oracle
  quantizers, float64 GEMMs, the same bf16 rounding points and activation):
  the GPU chain must agree with it (SQNR >= 35 dB between the two) and lose
  nothing against the float64 product of the unquantized inputs relative to
  it (within 0.5 dB).  On this workload the method itself stays below the
  25 dB single-linear bar for dx and the weight gradients (measured: out 24.1,
  dx 19.3, d_w1 16.8, d_w2 25.6, d_out_proj 24.8 dB): each 128-token block of
  the colwise (token-blocked) operands holds an outlier row 10-100x larger than
  the rest, which coarsens every other row of the block.  The silu * mul
  activation between the GEMMs is harness code (bf16 torch ops), as in the
  ToyModel.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import f32, gemm_max_err, lib
from mxfp8_precision_gemms_fp8bw_gb300 import inputs
from mxfp8_precision_gemms_fp8bw_gb300 import linear as L

pytestmark = pytest.mark.gpu
TOL = oracle.GEMM_TOL


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def _silu(t):
    return t * torch.sigmoid(t)


def test_ffn_step_parity_and_sqnr():
    t = inputs.ffn()
    x, w1, w2, wo, dy = (a.cuda() for a in (t.x, t.w1, t.w2, t.out_proj, t.dy))
    q1, q2, qo = L.quantize_weight(w1), L.quantize_weight(w2), L.quantize_weight(wo)
    h1, _ = L.forward(x, q1)
    h2, _ = L.forward(x, q2)
    a = (_silu(h1.float()) * h2.float()).bfloat16()
    out, _ = L.forward(a, qo)
    da, d_wo = L.backward(dy, a, qo)
    sig = torch.sigmoid(h1.float())
    dh1 = (da.float() * h2.float() * (sig * (1 + h1.float() * (1 - sig)))).bfloat16()
    dh2 = (da.float() * _silu(h1.float())).bfloat16()
    dx1, d_w1 = L.backward(dh1, x, q1)
    dx2, d_w2 = L.backward(dh2, x, q2)
    dx = dx1.float() + dx2.float()
    torch.cuda.synchronize()

    # Element-wise parity of the GEMMs whose operands are the workload's inputs.
    xf, w1f, wof, dyf = f32(t.x), f32(t.w1), f32(t.out_proj), f32(t.dy)
    xq, xs = oracle.quant_1x128_row(xf)
    xd = oracle.dequant_1x128_row(xq, xs)
    wq, _, ws = oracle.quant_128x128(w1f)
    wd = oracle.dequant_128x128(wq, ws)
    assert gemm_max_err(f32(h1), xd @ wd.T, xd, wd) <= TOL
    dq, ds = oracle.quant_1x128_row(dyf)
    dd = oracle.dequant_1x128_row(dq, ds)
    oq, _, os_ = oracle.quant_128x128(wof)
    od = oracle.dequant_128x128(oq, os_)
    assert gemm_max_err(f32(da), dd @ od, dd, od.T) <= TOL

    gpu = {"out": f32(out), "dx": dx.cpu().numpy(), "d_w1": f32(d_w1), "d_w2": f32(d_w2), "d_out_proj": f32(d_wo)}
    chain = _oracle_chain(t)
    exact = _unquantized_chain(t)
    for k in gpu:
        assert oracle.sqnr_db(chain[k], gpu[k]) >= 35.0, k
        assert oracle.sqnr_db(exact[k], gpu[k]) >= oracle.sqnr_db(exact[k], chain[k]) - 0.5, k


def _bf(a):
    return torch.from_numpy(np.asarray(a, np.float32)).bfloat16().float().numpy()


def _oracle_chain(t):
    """The FFN step through the oracle, with the harness's bf16 rounding points."""
    x, w1, w2, wo, dy = (f32(v) for v in (t.x, t.w1, t.w2, t.out_proj, t.dy))

    def fwd(a, w):
        q, s = oracle.quant_1x128_row(a)
        wq, _, ws = oracle.quant_128x128(w)
        return oracle.gemm_fwd(q, s, wq, ws)

    def bwd(d, a, w):
        q, s = oracle.quant_1x128_row(d)
        wq, _, ws = oracle.quant_128x128(w)
        return oracle.gemm_dgrad(q, s, wq, ws), oracle.gemm_wgrad(*oracle.quant_1x128_col(d), *oracle.quant_1x128_col(a))

    h1, h2 = _bf(fwd(x, w1)), _bf(fwd(x, w2))
    s = 1.0 / (1.0 + np.exp(-h1.astype(np.float64)))
    a = _bf(h1 * s * h2)
    out = fwd(a, wo)
    da, d_wo = bwd(dy, a, wo)
    da = _bf(da)
    dh1, dh2 = _bf(da * h2 * (s * (1 + h1 * (1 - s)))), _bf(da * h1 * s)
    dx1, d_w1 = bwd(dh1, x, w1)
    dx2, d_w2 = bwd(dh2, x, w2)
    return {"out": out, "dx": dx1 + dx2, "d_w1": d_w1, "d_w2": d_w2, "d_out_proj": d_wo}


def _unquantized_chain(t):
    X, W1, W2, WO, DY = (f32(v).astype(np.float64) for v in (t.x, t.w1, t.w2, t.out_proj, t.dy))
    H1, H2 = X @ W1.T, X @ W2.T
    S = 1.0 / (1.0 + np.exp(-H1))
    A = H1 * S * H2
    DA = DY @ WO
    DH1 = DA * H2 * (S * (1 + H1 * (1 - S)))
    DH2 = DA * H1 * S
    return {"out": A @ WO.T, "dx": DH1 @ W1 + DH2 @ W2, "d_w1": DH1.T @ X, "d_w2": DH2.T @ X, "d_out_proj": DY.T @ A}


@pytest.mark.parametrize("which", [0, 1])
def test_large_token_linear_full_size_sampled(which):
    t = inputs.large(which)
    M, K = t.x.shape
    N = t.w.shape[0]
    x, w, dy = t.x.cuda(), t.w.cuda(), t.dy.cuda()
    wq = L.quantize_weight(w)
    y, _ = L.forward(x, wq)
    dx, dW = L.backward(dy, x, wq)
    torch.cuda.synchronize()
    rng = np.random.default_rng(which)
    rows = np.sort(rng.choice(M, 128, replace=False))
    xf, wf, dyf = f32(t.x[rows]), f32(t.w), f32(t.dy[rows])
    wq_, _, ws_ = oracle.quant_128x128(wf)
    wd = oracle.dequant_128x128(wq_, ws_)
    xd = oracle.dequant_1x128_row(*oracle.quant_1x128_row(xf))
    assert gemm_max_err(f32(y[rows]), xd @ wd.T, xd, wd) <= TOL
    dd = oracle.dequant_1x128_row(*oracle.quant_1x128_row(dyf))
    assert gemm_max_err(f32(dx[rows]), dd @ wd, dd, wd.T) <= TOL
    # wgrad contracts over all 128000 tokens: sampled rows n and columns k
    ns = np.sort(rng.choice(N, 128, replace=False))
    ks = np.sort(rng.choice(K, 128, replace=False))
    a = oracle.dequant_1x128_row(*oracle.quant_1x128_col(np.ascontiguousarray(f32(t.dy[:, ns]))))
    b = oracle.dequant_1x128_row(*oracle.quant_1x128_col(np.ascontiguousarray(f32(t.x[:, ks]))))
    assert gemm_max_err(f32(dW)[np.ix_(ns, ks)], a @ b.T, a, b) <= TOL
