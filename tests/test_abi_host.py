"""Host-side checks of the C ABI: the library builds, loads, exports exactly the
calls include/fp8bw.h declares, and rejects bad arguments with the documented
codes before touching any GPU (these run with no GPU present)."""
import ctypes
import os
import re

import pytest

from mxfp8_precision_gemms_fp8bw_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fp8bw.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_abi():
    names = _declared_functions()
    assert names == sorted([
        "fp8bw_quant_1x128_row", "fp8bw_quant_1x128_col", "fp8bw_quant_128x128", "fp8bw_quant_1x128_rowcol",
        "fp8bw_gemm_fwd", "fp8bw_gemm_fwd_quant", "fp8bw_gemm_dgrad", "fp8bw_gemm_wgrad", "fp8bw_gemm_wgrad_acc_f32",
        "fp8bw_gemm_wgrad_ws", "fp8bw_gemm_wgrad_workspace_bytes",
        "mxfp8_quant_1x32_row", "mxfp8_quant_1x32_col", "mxfp8_quant_3d_col", "mxfp8_quant_1x32_rowcol",
        "mxfp8_grouped_gemm",
        "mxfp8_grouped_gemm_workspace_bytes", "mxfp8_grouped_gemm_noalloc",
        "fp8bw_sync_status", "fp8bw_last_error", "fp8bw_selftest_bounded_wait",
    ])


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), name
    assert set(binding._SIGNATURES) == set(_declared_functions())


def test_library_is_sm103a_only_and_self_contained():
    path = build.LIB_PATH
    data = open(path, "rb").read()
    assert b"sm_103a" in data or b"sm_103" in data
    # static CUDA runtime: no libcudart dependency to resolve on the GPU machine
    import subprocess
    out = subprocess.run(["ldd", path], capture_output=True, text=True).stdout
    assert "libcudart" not in out


P = 1 << 20  # a fake, 16-byte aligned "device" address; never dereferenced


def test_dgrad_needs_wq_and_takes_wqT_optionally(L):
    # wq is required even when the transposed copy is given; wqT alone is not enough
    assert L.fp8bw_gemm_dgrad(P, 2 * P, None, 3 * P, 4 * P, 64 * P, 128, 256, 256, None) == binding.ERR_NULL
    assert L.fp8bw_gemm_dgrad(P, 2 * P, 3 * P, 5 * P + 8, 4 * P, 64 * P, 128, 256, 256, None) == binding.ERR_ALIGN
    assert L.fp8bw_gemm_dgrad(P, 2 * P, 3 * P + 8, None, 4 * P, 64 * P, 128, 256, 256, None) == binding.ERR_ALIGN


def test_null_pointers_rejected(L):
    assert L.fp8bw_quant_1x128_row(None, 128, 128, P, P * 2, None) == binding.ERR_NULL
    assert "non-NULL" in binding.last_error()
    assert L.fp8bw_gemm_fwd(P, P, None, P, P, 128, 256, 128, None) == binding.ERR_NULL
    assert L.mxfp8_grouped_gemm(0, P, P, P, P, None, 1, 32, 256, 128, P, 64 * P, 1 << 20, None) == binding.ERR_NULL
    assert L.mxfp8_grouped_gemm(0, P, P, P, P, P, 1, 32, 256, 128, P, None, 1 << 20, None) == binding.ERR_NULL


@pytest.mark.parametrize("R,C", [(0, 128), (128, 0), (100, 128), (128, 200), (-128, 128)])
def test_blockwise_shapes_rejected(L, R, C):
    assert L.fp8bw_quant_1x128_row(P, R, C, P * 64, P * 128, None) == binding.ERR_SHAPE
    assert L.fp8bw_quant_1x128_col(P, R, C, P * 64, P * 128, None) == binding.ERR_SHAPE
    assert L.fp8bw_quant_128x128(P, R, C, P * 64, None, P * 128, None) == binding.ERR_SHAPE


def test_gemm_shapes_rejected(L):
    # N must be a multiple of 256 for fwd (output columns), M/K of 128
    assert L.fp8bw_gemm_fwd(P, 2 * P, 3 * P, 4 * P, 64 * P, 128, 128, 128, None) == binding.ERR_SHAPE
    assert L.fp8bw_gemm_fwd(P, 2 * P, 3 * P, 4 * P, 64 * P, 96, 256, 128, None) == binding.ERR_SHAPE
    # dgrad: output columns are K
    assert L.fp8bw_gemm_dgrad(P, 2 * P, 3 * P, None, 4 * P, 64 * P, 128, 256, 384, None) == binding.ERR_SHAPE
    assert L.fp8bw_gemm_dgrad(P, 2 * P, 3 * P, 5 * P, 4 * P, 64 * P, 128, 256, 384, None) == binding.ERR_SHAPE
    # wgrad: contraction over M must be a multiple of 128
    assert L.fp8bw_gemm_wgrad(P, 2 * P, 3 * P, 4 * P, 64 * P, 64, 256, 256, None) == binding.ERR_SHAPE


def test_wgrad_accumulate_validation(L):
    assert L.fp8bw_gemm_wgrad_acc_f32(P, 2 * P, 3 * P, 4 * P, None, 128, 256, 256, None) == binding.ERR_NULL
    assert L.fp8bw_gemm_wgrad_acc_f32(P, 2 * P, 3 * P, 4 * P, 64 * P, 64, 256, 256, None) == binding.ERR_SHAPE
    assert L.fp8bw_gemm_wgrad_acc_f32(P, 2 * P, 3 * P, 4 * P, 64 * P, 128, 256, 128, None) == binding.ERR_SHAPE
    assert L.fp8bw_gemm_wgrad_acc_f32(P, 2 * P, 3 * P, 4 * P, 64 * P + 4, 128, 256, 256, None) == binding.ERR_ALIGN
    # the fp32 output is 4 bytes per element: [N, K] = 256 x 256 from P overlaps the operand at P + 1024
    assert L.fp8bw_gemm_wgrad_acc_f32(P + 1024, 2 * P, 3 * P, 4 * P, P, 128, 256, 256, None) == binding.ERR_LAYOUT


def test_fwd_quant_validation(L):
    ops = (P, 2 * P, 3 * P, 4 * P, 64 * P)                     # xq, xs, wq, ws, y
    dims = (128, 256, 128, None)                               # M, N, K, stream
    assert L.fp8bw_gemm_fwd_quant(*ops, None, 80 * P, None, None, *dims) == binding.ERR_NULL
    assert L.fp8bw_gemm_fwd_quant(*ops, 72 * P, 80 * P, 96 * P, None, *dims) == binding.ERR_NULL   # yqT without ysT
    assert L.fp8bw_gemm_fwd_quant(*ops, 72 * P + 8, 80 * P, None, None, *dims) == binding.ERR_ALIGN
    assert L.fp8bw_gemm_fwd_quant(*ops, 72 * P, 80 * P, 96 * P + 4, 104 * P, *dims) == binding.ERR_ALIGN
    # yq [128, 256] from 64P + 4096 overlaps y [128, 256] bf16 (64 KB from 64P)
    assert L.fp8bw_gemm_fwd_quant(*ops, 64 * P + 4096, 80 * P, None, None, *dims) == binding.ERR_LAYOUT
    assert L.fp8bw_gemm_fwd_quant(*ops, 72 * P, 80 * P, None, None, 128, 128, 128, None) == binding.ERR_SHAPE


def test_misaligned_pointers_rejected(L):
    assert L.fp8bw_quant_1x128_row(P + 8, 128, 128, 64 * P, 128 * P, None) == binding.ERR_ALIGN
    assert L.fp8bw_gemm_wgrad(P, 2 * P, 3 * P + 4, 4 * P, 64 * P, 128, 256, 256, None) == binding.ERR_ALIGN
    assert L.mxfp8_quant_1x32_row(P, 32, 32, 64 * P + 1, 128 * P, 0, None) == binding.ERR_ALIGN


def test_enum_arguments_rejected(L):
    assert L.mxfp8_quant_1x32_row(P, 32, 32, 64 * P, 128 * P, 2, None) == binding.ERR_ARG
    assert L.mxfp8_quant_3d_col(P, 2, 64, 64, 64 * P, 128 * P, -1, None) == binding.ERR_ARG
    assert L.mxfp8_grouped_gemm(3, P, 2 * P, 3 * P, 4 * P, 5 * P, 1, 32, 256, 128, 64 * P, 128 * P, 1 << 20,
                                None) == binding.ERR_ARG
    assert L.fp8bw_selftest_bounded_wait(0, None) == binding.ERR_ARG
    assert L.fp8bw_selftest_bounded_wait(3000000, None) == binding.ERR_ARG


def test_aliasing_outputs_rejected(L):
    # q overlapping x: a layout the kernels never take, reported instead of copied
    assert L.fp8bw_quant_1x128_row(P, 128, 128, P + 16, 128 * P, None) == binding.ERR_LAYOUT
    assert L.fp8bw_gemm_fwd(P, 2 * P, 3 * P, 4 * P, P, 128, 256, 128, None) == binding.ERR_LAYOUT


def test_valid_arguments_reach_the_device_check(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this checks the no-GPU path")
    rc = L.fp8bw_quant_1x128_row(P, 128, 128, 64 * P, 128 * P, None)
    assert rc == binding.ERR_UNSUPPORTED
    assert binding.last_error()


def test_binding_rejects_wrong_dtype_and_layout():
    import torch
    x = torch.zeros(128, 128, dtype=torch.float32)
    with pytest.raises(TypeError):
        binding._ptr(x, torch.bfloat16, "x")
    with pytest.raises(ValueError):
        binding._ptr(torch.zeros(128, 128, dtype=torch.bfloat16), torch.bfloat16, "x")  # CPU tensor


def test_grouped_workspace_size_is_host_only(L):
    n = L.mxfp8_grouped_gemm_workspace_bytes(0, 8, 16384, 8192, 5120)
    # FWD: A chunks (M/128 + G) x K/128, B chunks G*N/128 x K/128, 512 bytes each
    assert n == (136 * 40 + 512 * 40) * 512
    assert L.mxfp8_grouped_gemm_workspace_bytes(2, 8, 16384, 8192, 5120) == 136 * (64 + 40) * 512
    assert L.mxfp8_grouped_gemm_workspace_bytes(5, 8, 16384, 8192, 5120) == 0
    assert L.mxfp8_grouped_gemm_workspace_bytes(0, 8, 100, 8192, 5120) == 0


def test_grouped_rejects_small_or_misaligned_workspace(L):
    need = L.mxfp8_grouped_gemm_workspace_bytes(0, 2, 256, 256, 256)
    args = (0, P, 2 * P, 3 * P, 4 * P, 5 * P, 2, 256, 256, 256, 64 * P)
    assert L.mxfp8_grouped_gemm(*args, 128 * P, need - 1, None) == binding.ERR_ARG
    assert "workspace" in binding.last_error()
    assert L.mxfp8_grouped_gemm(*args, 128 * P + 16, need, None) == binding.ERR_ALIGN


def test_noalloc_rejects_dims_beyond_its_scratch(L):
    # DGRAD of 8 experts with K = N = 16384: ~33.6 MB of packed scales > 16 MiB
    need = L.mxfp8_grouped_gemm_workspace_bytes(1, 8, 16384, 16384, 16384)
    assert need > binding.NOALLOC_SCRATCH_BYTES
    rc = L.mxfp8_grouped_gemm_noalloc(1, P, 2 * P, 3 * P, 4 * P, 5 * P, 8, 16384, 16384, 16384, 64 * P, None)
    assert rc == binding.ERR_SHAPE
    assert "scratch" in binding.last_error()


def test_mx_rowcol_validation(L):
    # x [G=2, R=64, C=64] bf16 at P; q at 64P, e8 at 80P, qT at 96P, e8T at 112P
    args = (P, 2, 64, 64, 64 * P, 80 * P, 96 * P, 112 * P)
    assert L.mxfp8_quant_1x32_rowcol(P, 2, 64, 64, 64 * P, 80 * P, None, 112 * P, 0, None) == binding.ERR_NULL
    assert L.mxfp8_quant_1x32_rowcol(P, 2, 48, 64, 64 * P, 80 * P, 96 * P, 112 * P, 0, None) == binding.ERR_SHAPE
    assert L.mxfp8_quant_1x32_rowcol(P, 2, 64, 40, 64 * P, 80 * P, 96 * P, 112 * P, 0, None) == binding.ERR_SHAPE
    assert L.mxfp8_quant_1x32_rowcol(P, 0, 64, 64, 64 * P, 80 * P, 96 * P, 112 * P, 0, None) == binding.ERR_SHAPE
    assert L.mxfp8_quant_1x32_rowcol(P, 2, 64, 64, 64 * P, 80 * P + 4, 96 * P, 112 * P, 0, None) == binding.ERR_ALIGN
    assert L.mxfp8_quant_1x32_rowcol(*args, 2, None) == binding.ERR_ARG
    # qT overlapping q (8 KB of codes from 64P)
    assert L.mxfp8_quant_1x32_rowcol(P, 2, 64, 64, 64 * P, 80 * P, 64 * P + 4096, 112 * P, 0, None) == binding.ERR_LAYOUT
    # e8 overlapping x (16 KB of bf16 from P)
    assert L.mxfp8_quant_1x32_rowcol(P, 2, 64, 64, 64 * P, P + 1024, 96 * P, 112 * P, 0, None) == binding.ERR_LAYOUT
