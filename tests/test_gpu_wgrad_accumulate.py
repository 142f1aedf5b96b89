"""GPU parity of the fp32-accumulating wgrad, dW += dy^T x, through the C ABI.

* Against the float64 oracle (a float32 dW plus the oracle's 128_1_128_1
  GEMM): the output is fp32, so no bf16 rounding enters and the bar is the
  fp32 promotion error only (normalized 1e-4, same normalizer as the GEMM
  bar).
* Starting from zero, the fp32 result rounded to bf16 equals the bf16 wgrad
  output bit for bit (same kernel, same promotion order).
* Token-shard accumulation followed by an SGD step, the parity methodology of
  PR #4295 "Testing" (gradients after the expected reduction, parameter values
  after the optimizer step) on one GPU: the gradients of 128-aligned token
  shards, accumulated into one fp32 dW, match the full-batch gradient and the
  oracle, and so do the parameters after W -= lr * dW.  The SGD update itself
  is harness code (a torch op), as the optimizer is in the pages' tests.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import f32, gemm_max_err, lib
from mxfp8_precision_gemms_fp8bw_gb300 import binding as B

pytestmark = pytest.mark.gpu

ACC_TOL = 1e-4
FP32 = oracle.FP32_ROUNDOFF   # fp32 outputs: only fp32's own rounding is allowed on top of the bar


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def _bf16(rng, shape, scale):
    return torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32)).bfloat16()


def _gpu_col(t):
    qT, s = B.alloc_quant_1x128_col(t)
    B.fp8bw_quant_1x128_col(t, qT, s)
    return qT, s


def _oracle_wgrad(dy, x):
    a = oracle.quant_1x128_col(f32(dy))
    b = oracle.quant_1x128_col(f32(x))
    return oracle.gemm_wgrad(*a, *b), oracle.dequant_1x128_row(*a), oracle.dequant_1x128_row(*b)


@pytest.mark.parametrize("M,N,K,seed", [(128, 128, 256, 0), (512, 512, 768, 1), (1280, 384, 1024, 2)])
def test_wgrad_accumulate_matches_oracle(M, N, K, seed):
    rng = np.random.default_rng(100 + seed)
    x, dy = _bf16(rng, (M, K), 1.0), _bf16(rng, (M, N), 1e-3)
    dW0 = torch.from_numpy((rng.standard_normal((N, K)) * 1e-2).astype(np.float32))
    xd, dyd = x.cuda(), dy.cuda()
    dyqT, dysT = _gpu_col(dyd)
    xqT, xsT = _gpu_col(xd)
    dW = dW0.cuda()
    B.fp8bw_gemm_wgrad_acc_f32(dyqT, dysT, xqT, xsT, dW)
    B.fp8bw_sync_status()
    ref, a, b = _oracle_wgrad(dy, x)
    got = dW.cpu().numpy().astype(np.float64)
    assert gemm_max_err(got, dW0.numpy().astype(np.float64) + ref, a, b, FP32) <= ACC_TOL

    # From zero, rounding the fp32 result to bf16 reproduces the bf16 kernel.
    z = torch.zeros((N, K), dtype=torch.float32, device="cuda")
    B.fp8bw_gemm_wgrad_acc_f32(dyqT, dysT, xqT, xsT, z)
    dW_bf16 = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    B.fp8bw_gemm_wgrad(dyqT, dysT, xqT, xsT, dW_bf16)
    B.fp8bw_sync_status()
    assert torch.equal(z.bfloat16(), dW_bf16)


def test_token_shard_accumulation_and_sgd_step_parity():
    M, N, K = 1024, 256, 512
    rng = np.random.default_rng(7)
    x, dy = _bf16(rng, (M, K), 1.0), _bf16(rng, (M, N), 1e-3)
    w = _bf16(rng, (N, K), 0.02).float()
    xd, dyd = x.cuda(), dy.cuda()

    acc = torch.zeros((N, K), dtype=torch.float32, device="cuda")
    for lo, hi in ((0, 384), (384, 1024)):          # two 128-aligned token shards
        dyqT, dysT = _gpu_col(dyd[lo:hi].contiguous())
        xqT, xsT = _gpu_col(xd[lo:hi].contiguous())
        B.fp8bw_gemm_wgrad_acc_f32(dyqT, dysT, xqT, xsT, acc)
    full = torch.zeros((N, K), dtype=torch.float32, device="cuda")
    B.fp8bw_gemm_wgrad_acc_f32(*_gpu_col(dyd), *_gpu_col(xd), full)
    B.fp8bw_sync_status()

    ref, a, b = _oracle_wgrad(dy, x)
    got_acc, got_full = acc.cpu().numpy().astype(np.float64), full.cpu().numpy().astype(np.float64)
    # gradients: shard sum == full batch (fp32 summation order only) == oracle
    assert gemm_max_err(got_acc, got_full, a, b, FP32) <= 1e-5
    assert gemm_max_err(got_acc, ref, a, b, FP32) <= ACC_TOL

    # parameters after one SGD step
    lr = 0.5
    w_gpu = (w.cuda() - lr * acc).cpu().numpy().astype(np.float64)
    w_ref = w.numpy().astype(np.float64) - lr * ref
    assert gemm_max_err((w_gpu - w.numpy()) / lr, (w_ref - w.numpy()) / lr, a, b, FP32) <= ACC_TOL
