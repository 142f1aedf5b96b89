"""ctypes binding of libfp8bw.so: the C ABI's calls under the same names.

Argument marshalling only: each function takes torch CUDA tensors, checks
their dtype/device/contiguity, passes ``data_ptr()`` and the current CUDA
stream to the library, and raises ``Fp8bwError`` on a nonzero status.  Every
step of the computation runs in the library's kernels; there is no fallback.
``alloc_*`` helpers create output tensors of the shapes the ABI documents.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_LIB = None

OK = 0
ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_LAYOUT, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_ARG = range(1, 9)
MX_RCEIL, MX_FLOOR = 0, 1
GROUPED_FWD, GROUPED_DGRAD, GROUPED_WGRAD = 0, 1, 2

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int

_SIGNATURES = {
    "fp8bw_quant_1x128_row": [_P, _I64, _I64, _P, _P, _P],
    "fp8bw_quant_1x128_col": [_P, _I64, _I64, _P, _P, _P],
    "fp8bw_quant_128x128": [_P, _I64, _I64, _P, _P, _P, _P],
    "fp8bw_quant_1x128_rowcol": [_P, _I64, _I64, _P, _P, _P, _P, _P],
    "fp8bw_gemm_fwd": [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P],
    "fp8bw_gemm_fwd_quant": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P],
    "fp8bw_gemm_dgrad": [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P],
    "fp8bw_gemm_wgrad": [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P],
    "fp8bw_gemm_wgrad_acc_f32": [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P],
    "fp8bw_gemm_wgrad_ws": [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, ctypes.c_size_t, _P],
    "fp8bw_gemm_wgrad_workspace_bytes": [_I64, _I64, _I64],
    "mxfp8_quant_1x32_row": [_P, _I64, _I64, _P, _P, _INT, _P],
    "mxfp8_quant_1x32_col": [_P, _I64, _I64, _P, _P, _INT, _P],
    "mxfp8_quant_3d_col": [_P, _I64, _I64, _I64, _P, _P, _INT, _P],
    "mxfp8_quant_1x32_rowcol": [_P, _I64, _I64, _I64, _P, _P, _P, _P, _INT, _P],
    "mxfp8_grouped_gemm": [_INT, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, ctypes.c_size_t, _P],
    "mxfp8_grouped_gemm_workspace_bytes": [_INT, _I64, _I64, _I64, _I64],
    "mxfp8_grouped_gemm_noalloc": [_INT, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _P],
    "fp8bw_sync_status": [_P],
    "fp8bw_last_error": [],
    "fp8bw_selftest_bounded_wait": [ctypes.c_uint32, _P],
}


class Fp8bwError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"libfp8bw error {code}: {message}")
        self.code = code


def lib_path() -> str:
    return _build.LIB_PATH


def lib(build_if_missing: bool = False) -> ctypes.CDLL:
    """Loads libfp8bw.so (building it first if asked); raises if it is absent."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built; call mxfp8_precision_gemms_fp8bw_gb300.build.build()")
        handle = ctypes.CDLL(path)
        for name, args in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = {"fp8bw_last_error": ctypes.c_char_p,
                          "mxfp8_grouped_gemm_workspace_bytes": ctypes.c_size_t,
                          "fp8bw_gemm_wgrad_workspace_bytes": ctypes.c_size_t}.get(name, ctypes.c_int)
        _LIB = handle
    return _LIB


def last_error() -> str:
    return lib().fp8bw_last_error().decode()


def _check(rc: int) -> None:
    if rc != OK:
        raise Fp8bwError(rc, last_error())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None, dtype: torch.dtype, name: str):
    if t is None:
        return None
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous (row-major); the library never copies into a layout")
    return t.data_ptr()


_BF16, _U8, _F32, _I32 = torch.bfloat16, torch.uint8, torch.float32, torch.int32


def scale_ld_128x128(C: int) -> int:
    return (C // 128 + 3) // 4 * 4


# ------------------------------------------------------------------ quantizers

def fp8bw_quant_1x128_row(x, q, s, stream=None) -> None:
    R, C = x.shape
    _check(lib().fp8bw_quant_1x128_row(_ptr(x, _BF16, "x"), R, C, _ptr(q, _U8, "q"), _ptr(s, _F32, "s"), _stream(stream)))


def fp8bw_quant_1x128_col(x, qT, s, stream=None) -> None:
    R, C = x.shape
    _check(lib().fp8bw_quant_1x128_col(_ptr(x, _BF16, "x"), R, C, _ptr(qT, _U8, "qT"), _ptr(s, _F32, "s"), _stream(stream)))


def fp8bw_quant_1x128_rowcol(x, q, s, qT, sT, stream=None) -> None:
    R, C = x.shape
    _check(lib().fp8bw_quant_1x128_rowcol(_ptr(x, _BF16, "x"), R, C, _ptr(q, _U8, "q"), _ptr(s, _F32, "s"),
                                          _ptr(qT, _U8, "qT"), _ptr(sT, _F32, "sT"), _stream(stream)))


def fp8bw_quant_128x128(w, q, qT, s, stream=None) -> None:
    R, C = w.shape
    _check(lib().fp8bw_quant_128x128(_ptr(w, _BF16, "w"), R, C, _ptr(q, _U8, "q"), _ptr(qT, _U8, "qT"),
                                     _ptr(s, _F32, "s"), _stream(stream)))


def mxfp8_quant_1x32_row(x, q, e8, mode=MX_RCEIL, stream=None) -> None:
    R, C = x.shape
    _check(lib().mxfp8_quant_1x32_row(_ptr(x, _BF16, "x"), R, C, _ptr(q, _U8, "q"), _ptr(e8, _U8, "e8"), mode,
                                      _stream(stream)))


def mxfp8_quant_1x32_col(x, qT, e8, mode=MX_RCEIL, stream=None) -> None:
    R, C = x.shape
    _check(lib().mxfp8_quant_1x32_col(_ptr(x, _BF16, "x"), R, C, _ptr(qT, _U8, "qT"), _ptr(e8, _U8, "e8"), mode,
                                      _stream(stream)))


def mxfp8_quant_3d_col(w, qT, e8, mode=MX_RCEIL, stream=None) -> None:
    G, N, K = w.shape
    _check(lib().mxfp8_quant_3d_col(_ptr(w, _BF16, "w"), G, N, K, _ptr(qT, _U8, "qT"), _ptr(e8, _U8, "e8"), mode,
                                    _stream(stream)))


def mxfp8_quant_1x32_rowcol(x, q, e8, qT, e8T, mode=MX_RCEIL, stream=None) -> None:
    """Both MX quantizations of x [R, C] (G = 1) or of G stacked matrices
    x [G, R, C] from one read: q [G*R, C] / e8 [G*R, C/32] rowwise and
    qT [G, C, R] / e8T [G, C, R/32] colwise (qT [C, R], e8T [C, R/32] for 2D x)."""
    G, R, C = (1, *x.shape) if x.dim() == 2 else x.shape
    _check(lib().mxfp8_quant_1x32_rowcol(_ptr(x, _BF16, "x"), G, R, C, _ptr(q, _U8, "q"), _ptr(e8, _U8, "e8"),
                                         _ptr(qT, _U8, "qT"), _ptr(e8T, _U8, "e8T"), mode, _stream(stream)))


# ------------------------------------------------------------------ GEMMs

def fp8bw_gemm_fwd(xq, xs, wq, ws, y, stream=None) -> None:
    M, K = xq.shape
    N = wq.shape[0]
    _check(lib().fp8bw_gemm_fwd(_ptr(xq, _U8, "xq"), _ptr(xs, _F32, "xs"), _ptr(wq, _U8, "wq"), _ptr(ws, _F32, "ws"),
                                _ptr(y, _BF16, "y"), M, N, K, _stream(stream)))


def fp8bw_gemm_fwd_quant(xq, xs, wq, ws, y, yq, ys, yqT=None, ysT=None, stream=None) -> None:
    M, K = xq.shape
    N = wq.shape[0]
    _check(lib().fp8bw_gemm_fwd_quant(_ptr(xq, _U8, "xq"), _ptr(xs, _F32, "xs"), _ptr(wq, _U8, "wq"),
                                      _ptr(ws, _F32, "ws"), _ptr(y, _BF16, "y"), _ptr(yq, _U8, "yq"),
                                      _ptr(ys, _F32, "ys"), _ptr(yqT, _U8, "yqT"), _ptr(ysT, _F32, "ysT"), M, N, K,
                                      _stream(stream)))


def fp8bw_gemm_dgrad(dyq, dys, wq, wqT, ws, dx, stream=None) -> None:
    """dx = dy W from W's codes wq [N, K]; wqT [K, N] (its transposed copy) is optional."""
    M, N = dyq.shape
    K = wq.shape[1]
    _check(lib().fp8bw_gemm_dgrad(_ptr(dyq, _U8, "dyq"), _ptr(dys, _F32, "dys"), _ptr(wq, _U8, "wq"),
                                  _ptr(wqT, _U8, "wqT"), _ptr(ws, _F32, "ws"), _ptr(dx, _BF16, "dx"), M, N, K,
                                  _stream(stream)))


def fp8bw_gemm_wgrad(dyqT, dysT, xqT, xsT, dW, stream=None) -> None:
    N, M = dyqT.shape
    K = xqT.shape[0]
    _check(lib().fp8bw_gemm_wgrad(_ptr(dyqT, _U8, "dyqT"), _ptr(dysT, _F32, "dysT"), _ptr(xqT, _U8, "xqT"),
                                  _ptr(xsT, _F32, "xsT"), _ptr(dW, _BF16, "dW"), M, N, K, _stream(stream)))


def fp8bw_gemm_wgrad_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().fp8bw_gemm_wgrad_workspace_bytes(M, N, K))


def alloc_wgrad_workspace(M: int, N: int, K: int, device) -> torch.Tensor | None:
    """The workspace fp8bw_gemm_wgrad_ws wants for these dims on this device, or None if it needs none."""
    n = fp8bw_gemm_wgrad_workspace_bytes(M, N, K)
    return torch.empty(n, dtype=_U8, device=device) if n else None


def fp8bw_gemm_wgrad_ws(dyqT, dysT, xqT, xsT, dW, workspace, stream=None) -> None:
    N, M = dyqT.shape
    K = xqT.shape[0]
    ws = _ptr(workspace, _U8, "workspace") if workspace is not None else None
    nbytes = workspace.numel() if workspace is not None else 0
    _check(lib().fp8bw_gemm_wgrad_ws(_ptr(dyqT, _U8, "dyqT"), _ptr(dysT, _F32, "dysT"), _ptr(xqT, _U8, "xqT"),
                                     _ptr(xsT, _F32, "xsT"), _ptr(dW, _BF16, "dW"), M, N, K, ws, nbytes,
                                     _stream(stream)))


def fp8bw_gemm_wgrad_acc_f32(dyqT, dysT, xqT, xsT, dW, stream=None) -> None:
    """dW (fp32 [N, K]) += dy^T x."""
    N, M = dyqT.shape
    K = xqT.shape[0]
    _check(lib().fp8bw_gemm_wgrad_acc_f32(_ptr(dyqT, _U8, "dyqT"), _ptr(dysT, _F32, "dysT"), _ptr(xqT, _U8, "xqT"),
                                          _ptr(xsT, _F32, "xsT"), _ptr(dW, _F32, "dW"), M, N, K, _stream(stream)))


def mxfp8_grouped_gemm_workspace_bytes(kind, G, M, N, K) -> int:
    return int(lib().mxfp8_grouped_gemm_workspace_bytes(int(kind), G, M, N, K))


def alloc_grouped_workspace(kind, G, M, N, K, device) -> torch.Tensor:
    """A uint8 device buffer large enough for mxfp8_grouped_gemm's packed scales."""
    n = mxfp8_grouped_gemm_workspace_bytes(kind, G, M, N, K)
    if n == 0:
        raise Fp8bwError(ERR_SHAPE, "invalid grouped GEMM dims")
    return torch.empty(n, dtype=_U8, device=device)


def mxfp8_grouped_gemm(kind, a, a_e8, b, b_e8, group_end, G, M, N, K, out, workspace, stream=None) -> None:
    _check(lib().mxfp8_grouped_gemm(int(kind), _ptr(a, _U8, "a"), _ptr(a_e8, _U8, "a_e8"), _ptr(b, _U8, "b"),
                                    _ptr(b_e8, _U8, "b_e8"), _ptr(group_end, _I32, "group_end"), G, M, N, K,
                                    _ptr(out, _BF16, "out"), _ptr(workspace, _U8, "workspace"),
                                    workspace.numel(), _stream(stream)))


NOALLOC_SCRATCH_BYTES = 16 << 20


def mxfp8_grouped_gemm_noalloc(kind, a, a_e8, b, b_e8, group_end, G, M, N, K, out, stream=None) -> None:
    """mxfp8_grouped_gemm without a workspace argument: for callers that cannot
    allocate device memory, the library uses its own fixed 16 MiB array."""
    _check(lib().mxfp8_grouped_gemm_noalloc(int(kind), _ptr(a, _U8, "a"), _ptr(a_e8, _U8, "a_e8"), _ptr(b, _U8, "b"),
                                            _ptr(b_e8, _U8, "b_e8"), _ptr(group_end, _I32, "group_end"), G, M, N, K,
                                            _ptr(out, _BF16, "out"), _stream(stream)))


def fp8bw_sync_status(stream=None) -> None:
    _check(lib().fp8bw_sync_status(_stream(stream)))


def fp8bw_selftest_bounded_wait(timeout_us: int, stream=None) -> None:
    _check(lib().fp8bw_selftest_bounded_wait(int(timeout_us), _stream(stream)))


# ------------------------------------------------------------------ output allocation helpers

def alloc_quant_1x128_row(x: torch.Tensor):
    R, C = x.shape
    return (torch.empty((R, C), dtype=_U8, device=x.device), torch.empty((C // 128, R), dtype=_F32, device=x.device))


def alloc_quant_1x128_col(x: torch.Tensor):
    R, C = x.shape
    return (torch.empty((C, R), dtype=_U8, device=x.device), torch.empty((R // 128, C), dtype=_F32, device=x.device))


def alloc_quant_128x128(w: torch.Tensor, with_transpose: bool = True):
    R, C = w.shape
    q = torch.empty((R, C), dtype=_U8, device=w.device)
    qT = torch.empty((C, R), dtype=_U8, device=w.device) if with_transpose else None
    s = torch.zeros((R // 128, scale_ld_128x128(C)), dtype=_F32, device=w.device)
    return q, qT, s


def alloc_mx_row(x: torch.Tensor):
    R, C = x.shape
    return (torch.empty((R, C), dtype=_U8, device=x.device), torch.empty((R, C // 32), dtype=_U8, device=x.device))


def alloc_mx_col(x: torch.Tensor):
    R, C = x.shape
    return (torch.empty((C, R), dtype=_U8, device=x.device), torch.empty((C, R // 32), dtype=_U8, device=x.device))


def alloc_mx_3d_col(w: torch.Tensor):
    G, N, K = w.shape
    return (torch.empty((G, K, N), dtype=_U8, device=w.device), torch.empty((G, K, N // 32), dtype=_U8, device=w.device))
