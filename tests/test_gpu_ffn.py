"""The toy FFN workload (PR #4295's ToyModel: w1, w2 up-projections and
out_proj, tokens 4096, dim 2048, hidden 8192, 1 % outlier rows in x) forward
and backward through Float8BlockwiseLinear GEMMs, and the large-token dense
workloads (M = 128000) whose wgrad contracts over 128000 tokens.

* Every one of the FFN step's nine GEMMs is checked against the oracle element
  by element (normalized error <= 2e-3), each fed the bf16 tensors the GPU step
  itself produced (x, a, dy, dh1, dh2 and the weights), quantized by the
  oracle; the library's quantizations of those intermediates are checked byte
  for byte.
* The whole FFN step is run a second time through the oracle (oracle
  quantizers, float64 GEMMs, the same bf16 rounding points and activation):
  the GPU chain must agree with it (SQNR >= 35 dB between the two) and lose
  nothing against the float64 product of the unquantized inputs relative to
  it (within 0.5 dB).  On this workload the method itself stays below the
  25 dB single-linear bar for dx and the weight gradients (measured: out 24.1,
  dx 19.3, d_w1 16.8, d_w2 25.6, d_out_proj 24.8 dB): each 128-token block of
  the colwise (token-blocked) operands holds an outlier row 10-100x larger than
  the rest, which coarsens every other row of the block.  The silu * mul
  activation between the GEMMs is the model's own code, the bf16 torch ops
  autograd runs for silu(h1) * h2 (each op's result rounded to bf16).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import bits, f32, gemm_max_err, lib, u8
from mxfp8_precision_gemms_fp8bw_gb300 import inputs
from mxfp8_precision_gemms_fp8bw_gb300 import linear as L

pytestmark = pytest.mark.gpu
TOL = oracle.GEMM_TOL


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def _fwd_ref(a, w):
    """Oracle y = a w^T on bf16-valued float32 inputs, with the dequantized operands."""
    q, s = oracle.quant_1x128_row(a)
    wq, _, ws = oracle.quant_128x128(w)
    ad, wd = oracle.dequant_1x128_row(q, s), oracle.dequant_128x128(wq, ws)
    return ad @ wd.T, ad, wd


def _dgrad_ref(d, w):
    q, s = oracle.quant_1x128_row(d)
    wq, _, ws = oracle.quant_128x128(w)
    dd, wd = oracle.dequant_1x128_row(q, s), oracle.dequant_128x128(wq, ws)
    return dd @ wd, dd, wd.T


def _wgrad_ref(d, a):
    dq, ds = oracle.quant_1x128_col(d)
    aq, as_ = oracle.quant_1x128_col(a)
    dd, ad = oracle.dequant_1x128_row(dq, ds), oracle.dequant_1x128_row(aq, as_)
    return dd @ ad.T, dd, ad


def test_ffn_step_parity_and_sqnr():
    t = inputs.ffn()
    x, w1, w2, wo, dy = (v.cuda() for v in (t.x, t.w1, t.w2, t.out_proj, t.dy))
    M, D = t.x.shape
    H = t.w1.shape[0]
    step = L.ToyFFNStep(M, D, H, device=x.device)
    res = step.step(x, w1, w2, wo, dy)
    torch.cuda.synchronize()

    xf, w1f, w2f, wof, dyf = (f32(v) for v in (t.x, t.w1, t.w2, t.out_proj, t.dy))
    af, dh1f, dh2f = f32(step.a), f32(step.dh1), f32(step.dh2)

    # The library's quantizations of the step's own intermediates, byte for byte.
    for src, q in ((af, step.aa), (dh1f, step.dh1a), (dh2f, step.dh2a)):
        qo, so = oracle.quant_1x128_row(src)
        assert np.array_equal(u8(q["q"]), qo) and np.array_equal(bits(q["s"]), bits(so))
        qTo, sTo = oracle.quant_1x128_col(src)
        assert np.array_equal(u8(q["qT"]), qTo) and np.array_equal(bits(q["sT"]), bits(sTo))

    # All nine GEMMs, element by element, each on the GPU step's own inputs.
    cases = {
        "fwd w1 (h1)": (f32(step.h1), _fwd_ref(xf, w1f)),
        "fwd w2 (h2)": (f32(step.h2), _fwd_ref(xf, w2f)),
        "fwd out_proj (out)": (f32(step.out), _fwd_ref(af, wof)),
        "dgrad out_proj (da)": (f32(step.da), _dgrad_ref(dyf, wof)),
        "wgrad out_proj": (f32(step.d_wo), _wgrad_ref(dyf, af)),
        "dgrad w1 (dx1)": (f32(step.dx1), _dgrad_ref(dh1f, w1f)),
        "wgrad w1": (f32(step.d_w1), _wgrad_ref(dh1f, xf)),
        "dgrad w2 (dx2)": (f32(step.dx2), _dgrad_ref(dh2f, w2f)),
        "wgrad w2": (f32(step.d_w2), _wgrad_ref(dh2f, xf)),
    }
    for name, (got, (ref, an, bn)) in cases.items():
        assert gemm_max_err(got, ref, an, bn) <= TOL, name

    gpu = {"out": f32(res["out"]), "dx": f32(step.dx1).astype(np.float64) + f32(step.dx2),
           "d_w1": f32(res["d_w1"]), "d_w2": f32(res["d_w2"]), "d_out_proj": f32(res["d_out_proj"])}
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
    s1 = _bf(h1 * s)  # silu(h1) in bf16
    a = _bf(s1 * h2)
    out = fwd(a, wo)
    da, d_wo = bwd(dy, a, wo)
    da = _bf(da)
    g = _bf(da * h2)  # the gradient reaching silu's output
    dh1, dh2 = _bf(g * (s * (1 + h1 * (1 - s)))), _bf(da * s1)
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
