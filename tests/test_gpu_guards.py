"""Guard canaries around every output: each call must write exactly its output
region and nothing before or after it (the role compute-sanitizer's memcheck
would play; it is not available on this machine).  Covers the quantizers, the
three blockwise GEMMs and the grouped GEMM, including the long-contraction
wgrad shape class that crashed the prior art (PR #2386, torchtitan bullet)."""
import numpy as np
import pytest
import torch

from gpu_util import lib
from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
from mxfp8_precision_gemms_fp8bw_gb300 import inputs

pytestmark = pytest.mark.gpu

GUARD = 4096
CANARY = 0xA5


class Guarded:
    """A device buffer with GUARD canary bytes on both sides of the payload."""

    def __init__(self, shape, dtype):
        self.nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((self.nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def intact(self) -> bool:
        r = self.raw.cpu().numpy()
        return bool(np.all(r[:GUARD] == CANARY) and np.all(r[GUARD + self.nbytes:] == CANARY))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def test_quantizer_outputs_stay_in_bounds():
    x = inputs.linear_inputs(384, 640, 256, seed=5).x.cuda()
    R, C = x.shape
    q, s = Guarded((R, C), torch.uint8), Guarded((C // 128, R), torch.float32)
    B.fp8bw_quant_1x128_row(x, q.t, s.t)
    qT, sT = Guarded((C, R), torch.uint8), Guarded((R // 128, C), torch.float32)
    B.fp8bw_quant_1x128_col(x, qT.t, sT.t)
    wq, wqT, ws = Guarded((R, C), torch.uint8), Guarded((C, R), torch.uint8), Guarded((R // 128, B.scale_ld_128x128(C)), torch.float32)
    B.fp8bw_quant_128x128(x, wq.t, wqT.t, ws.t)
    mq, me = Guarded((R, C), torch.uint8), Guarded((R, C // 32), torch.uint8)
    B.mxfp8_quant_1x32_row(x, mq.t, me.t)
    mqT, meT = Guarded((C, R), torch.uint8), Guarded((C, R // 32), torch.uint8)
    B.mxfp8_quant_1x32_col(x, mqT.t, meT.t)
    B.fp8bw_sync_status()
    for g in (q, s, qT, sT, wq, wqT, ws, mq, me, mqT, meT):
        assert g.intact()


@pytest.mark.parametrize("M,N,K", [(256, 512, 256), (2048, 256, 512)])
def test_gemm_outputs_stay_in_bounds(M, N, K):
    t = inputs.linear_inputs(M, K, N, seed=M)
    x, w, dy = t.x.cuda(), t.w.cuda(), t.dy.cuda()
    xq, xs = B.alloc_quant_1x128_row(x)
    B.fp8bw_quant_1x128_row(x, xq, xs)
    wq, wqT, ws = B.alloc_quant_128x128(w)
    B.fp8bw_quant_128x128(w, wq, wqT, ws)
    dyq, dys = B.alloc_quant_1x128_row(dy)
    B.fp8bw_quant_1x128_row(dy, dyq, dys)
    dyqT, dysT = B.alloc_quant_1x128_col(dy)
    B.fp8bw_quant_1x128_col(dy, dyqT, dysT)
    xqT, xsT = B.alloc_quant_1x128_col(x)
    B.fp8bw_quant_1x128_col(x, xqT, xsT)
    y, dx, dW = Guarded((M, N), torch.bfloat16), Guarded((M, K), torch.bfloat16), Guarded((N, K), torch.bfloat16)
    B.fp8bw_gemm_fwd(xq, xs, wq, ws, y.t)
    B.fp8bw_gemm_dgrad(dyq, dys, wq, wqT, ws, dx.t)
    B.fp8bw_gemm_wgrad(dyqT, dysT, xqT, xsT, dW.t)
    B.fp8bw_sync_status()
    assert y.intact() and dx.intact() and dW.intact()


def test_grouped_outputs_stay_in_bounds():
    rng = np.random.default_rng(3)
    M, K, N, G = 384, 256, 512, 3
    ge = torch.tensor([96, 96, 384], dtype=torch.int32, device="cuda")
    x = inputs.normal_bf16(rng, (M, K), 1.0).cuda()
    w = inputs.normal_bf16(rng, (G, N, K), 0.02).cuda()
    xq, xe = B.alloc_mx_row(x)
    B.mxfp8_quant_1x32_row(x, xq, xe)
    wq, we = B.alloc_mx_row(w.view(G * N, K))
    B.mxfp8_quant_1x32_row(w.view(G * N, K), wq, we)
    y = Guarded((M, N), torch.bfloat16)
    n = B.mxfp8_grouped_gemm_workspace_bytes(B.GROUPED_FWD, G, M, N, K)
    ws = Guarded((n,), torch.uint8)
    assert ws.t.data_ptr() % 256 == 0
    B.mxfp8_grouped_gemm(B.GROUPED_FWD, xq, xe, wq, we, ge, G, M, N, K, y.t, ws.t)
    B.fp8bw_sync_status()
    assert y.intact() and ws.intact()
