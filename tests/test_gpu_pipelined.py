"""The pipelined host-to-host step runner (uploads, kernels and downloads of
neighbouring steps on three streams, two device buffer sets) returns, for every
step, exactly what the plain step returns on the same inputs: the overlap
changes when work runs, not what it computes."""
import pytest
import torch

from gpu_util import lib
from mxfp8_precision_gemms_fp8bw_gb300 import linear as L

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def test_pipelined_steps_equal_plain_steps():
    M, N, K, steps = 384, 512, 768, 5
    g = torch.Generator().manual_seed(7)
    host = lambda shape, s: (torch.randn(shape, generator=g) * s).bfloat16().pin_memory()  # noqa: E731
    ins = [(host((M, K), 1.0), host((N, K), 0.02), host((M, N), 1e-3)) for _ in range(steps)]
    outs = [tuple(torch.empty(shape, dtype=torch.bfloat16).pin_memory() for shape in ((M, N), (M, K), (N, K)))
            for _ in range(steps)]
    pipe = L.PipelinedLinearSteps(M, N, K)
    for (x_h, w_h, dy_h), (y_h, dx_h, dW_h) in zip(ins, outs):
        pipe.step(x_h, w_h, dy_h, y_h, dx_h, dW_h)
    pipe.synchronize()

    ws = L.BlockwiseLinearWorkspace(M, N, K)
    for (x_h, w_h, dy_h), got in zip(ins, outs):
        want = ws.step(x_h.cuda(), w_h.cuda(), dy_h.cuda())
        torch.cuda.synchronize()
        for g_, w_ in zip(got, want):
            assert torch.equal(g_, w_.cpu())


def test_pipelined_rejects_pageable_host_buffers():
    M, N, K = 128, 256, 256
    pipe = L.PipelinedLinearSteps(M, N, K)
    bf = torch.bfloat16
    args = [torch.zeros(s, dtype=bf) for s in ((M, K), (N, K), (M, N), (M, N), (M, K), (N, K))]
    with pytest.raises(ValueError):
        pipe.step(*args)
