"""The library's calls can be captured in a CUDA graph: the six calls of a
blockwise linear step and the MXFP8 grouped forward, captured once and
replayed on new inputs, give exactly what eager calls give."""
import numpy as np
import pytest
import torch

from gpu_util import lib
from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
from mxfp8_precision_gemms_fp8bw_gb300 import inputs
from mxfp8_precision_gemms_fp8bw_gb300 import linear as L

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def test_blockwise_step_graph_replay_equals_eager():
    M, N, K = 384, 512, 768
    a = inputs.linear_inputs(M, K, N, seed=21)
    b = inputs.linear_inputs(M, K, N, seed=22)
    x, w, dy = a.x.cuda(), a.w.cuda(), a.dy.cuda()
    ws = L.BlockwiseLinearWorkspace(M, N, K)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ws.step(x, w, dy, stream=s)  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ws.step(x, w, dy)
    for t in (b, a):
        x.copy_(t.x.cuda()), w.copy_(t.w.cuda()), dy.copy_(t.dy.cuda())
        g.replay()
        torch.cuda.synchronize()
        got = [o.clone() for o in (ws.y, ws.dx, ws.dW)]
        eager = L.BlockwiseLinearWorkspace(M, N, K)
        want = eager.step(t.x.cuda(), t.w.cuda(), t.dy.cuda())
        torch.cuda.synchronize()
        B.fp8bw_sync_status()
        for g_, w_ in zip(got, want):
            assert torch.equal(g_, w_)


def test_mx_grouped_forward_graph_replay_equals_eager():
    rng = np.random.default_rng(23)
    M, K, N, G = 256, 256, 256, 3
    ge = torch.from_numpy(np.array([96, 160, 256], np.int32)).cuda()
    x = (torch.randn(M, K, device="cuda") ).bfloat16()
    w = (0.02 * torch.randn(G, N, K, device="cuda")).bfloat16()
    wq = L.mx_quantize_experts(w)
    xq, xe = B.alloc_mx_row(x)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    wsp = B.alloc_grouped_workspace(B.GROUPED_FWD, G, M, N, K, x.device)

    def fwd():
        B.mxfp8_quant_1x32_row(x, xq, xe)
        B.mxfp8_grouped_gemm(B.GROUPED_FWD, xq, xe, wq.q_row, wq.e8_row, ge, G, M, N, K, y, wsp)

    fwd()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fwd()
    x.copy_(torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).bfloat16().cuda())
    g.replay()
    torch.cuda.synchronize()
    got = y.clone()
    want = L.mx_moe_forward(x, wq, ge)
    torch.cuda.synchronize()
    B.fp8bw_sync_status()
    assert torch.equal(got, want)
