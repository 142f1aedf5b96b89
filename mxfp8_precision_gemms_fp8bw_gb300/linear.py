"""Float8BlockwiseLinear and the MXFP8 MoE linear as sequences of libfp8bw calls.

PR #4295 ("add FSDP and TP tests for Float8BlockwiseLinear", Summary) names a
drop-in ``nn.Linear`` replacement whose forward is one blockwise-scaled GEMM
and whose backward is two; PR #2386 (description) gives the block shapes.
This module only orders the library calls and allocates their outputs with
torch; every quantization and GEMM runs in libfp8bw's kernels.

Forward   : x -> 1x128 rowwise and colwise in one pass (q_x, s_x, q_x^T, s_x^T);
            W -> 128x128 (q_W, s_W); y = gemm_fwd(q_x, s_x, q_W, s_W).
            The colwise x codes (1 byte per element) are kept for backward
            instead of the bf16 x.
Backward  : dy -> 1x128 rowwise and colwise in one pass;
            dx = gemm_dgrad(q_dy, s_dy, q_W, s_W) (W's codes read transposed by the
            tensor core); dW = gemm_wgrad(q_dy^T, s_dy^T, q_x^T, s_x^T)
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as B


@dataclass
class QuantizedWeight:
    q: torch.Tensor                # e4m3 [N, K]
    qT: torch.Tensor | None        # e4m3 [K, N], the same codes transposed, or None
    s: torch.Tensor                # fp32 [N/128][LD(K)]


def quantize_weight(w: torch.Tensor, stream=None, with_transpose: bool = False) -> QuantizedWeight:
    """128x128 quantization of W.  dgrad reads q itself (transposed by the
    tensor core), so the transposed copy is written only when asked for."""
    q, qT, s = B.alloc_quant_128x128(w, with_transpose=with_transpose)
    B.fp8bw_quant_128x128(w, q, qT, s, stream)
    return QuantizedWeight(q, qT, s)


def forward(x: torch.Tensor, wq: QuantizedWeight, stream=None):
    """y = x W^T.  Returns y and the colwise codes of x (q_x^T, s_x^T) that
    the backward pass needs, both quantizations coming from one read of x."""
    M, K = x.shape
    N = wq.q.shape[0]
    xq, xs = B.alloc_quant_1x128_row(x)
    xqT, xsT = B.alloc_quant_1x128_col(x)
    B.fp8bw_quant_1x128_rowcol(x, xq, xs, xqT, xsT, stream)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    B.fp8bw_gemm_fwd(xq, xs, wq.q, wq.s, y, stream)
    return y, (xqT, xsT)


def backward(dy: torch.Tensor, x_col, wq: QuantizedWeight, stream=None, dW_acc: torch.Tensor | None = None):
    """dx = dy W and dW = dy^T x.  x_col is (q_x^T, s_x^T) from forward, or
    the bf16 x itself (then quantized colwise here).  Returns (dx, dW); with
    an fp32 ``dW_acc`` [N, K] the gradient is added to it instead (gradient
    accumulation) and dW_acc is returned as dW."""
    M, N = dy.shape
    if isinstance(x_col, torch.Tensor):
        xqT, xsT = B.alloc_quant_1x128_col(x_col)
        B.fp8bw_quant_1x128_col(x_col, xqT, xsT, stream)
    else:
        xqT, xsT = x_col
    K = xqT.shape[0]
    dyq, dys = B.alloc_quant_1x128_row(dy)
    dyqT, dysT = B.alloc_quant_1x128_col(dy)
    B.fp8bw_quant_1x128_rowcol(dy, dyq, dys, dyqT, dysT, stream)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=dy.device)
    B.fp8bw_gemm_dgrad(dyq, dys, wq.q, wq.qT, wq.s, dx, stream)
    if dW_acc is not None:
        B.fp8bw_gemm_wgrad_acc_f32(dyqT, dysT, xqT, xsT, dW_acc, stream)
        return dx, dW_acc
    dW = torch.empty((N, K), dtype=torch.bfloat16, device=dy.device)
    B.fp8bw_gemm_wgrad_ws(dyqT, dysT, xqT, xsT, dW, B.alloc_wgrad_workspace(M, N, K, dy.device), stream)
    return dx, dW


class _Float8BlockwiseLinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, w):
        wq = quantize_weight(w)
        y, x_col = forward(x, wq)
        ctx.x_col = x_col
        ctx.wq = wq
        return y

    @staticmethod
    def backward(ctx, dy):
        dx, dW = backward(dy.contiguous(), ctx.x_col, ctx.wq)
        return dx, dW


class Float8BlockwiseLinear(torch.nn.Module):
    """nn.Linear without bias whose three GEMMs run blockwise-scaled in e4m3.

    Inputs are 2D bf16 CUDA tensors [tokens, in_features]; in_features,
    out_features and tokens must be multiples of 128, and the output column
    count of each GEMM (out_features for forward, in_features for both
    gradients) a multiple of 256.
    """

    def __init__(self, in_features: int, out_features: int, device=None):
        super().__init__()
        self.weight = torch.nn.Parameter(torch.empty((out_features, in_features), dtype=torch.bfloat16, device=device))
        torch.nn.init.normal_(self.weight, std=0.02)

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return _Float8BlockwiseLinearFn.apply(x, self.weight)


# ------------------------------------------------------------------ MXFP8 MoE linear

@dataclass
class MxExpertWeights:
    q_row: torch.Tensor    # e4m3 [G, N, K], 1x32 along K (forward)
    e8_row: torch.Tensor   # [G*N, K/32]
    qT_col: torch.Tensor   # e4m3 [G, K, N], 1x32 along N (dgrad, 3D colwise)
    e8_col: torch.Tensor   # [G, K, N/32]


def mx_quantize_experts(w: torch.Tensor, mode: int = B.MX_RCEIL, stream=None) -> MxExpertWeights:
    """Rowwise (forward) and 3D colwise (dgrad) MX codes of the expert
    weights w [G, N, K], both from one read of w."""
    G, N, K = w.shape
    q, e8 = B.alloc_mx_row(w.view(G * N, K))
    qT, e8c = B.alloc_mx_3d_col(w)
    B.mxfp8_quant_1x32_rowcol(w, q, e8, qT, e8c, mode, stream)
    return MxExpertWeights(q.view(G, N, K), e8, qT, e8c)


def mx_moe_forward(x: torch.Tensor, wq: MxExpertWeights, group_end: torch.Tensor, mode: int = B.MX_RCEIL, stream=None):
    M, K = x.shape
    G, N, _ = wq.q_row.shape
    xq, xe = B.alloc_mx_row(x)
    B.mxfp8_quant_1x32_row(x, xq, xe, mode, stream)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws = B.alloc_grouped_workspace(B.GROUPED_FWD, G, M, N, K, x.device)
    B.mxfp8_grouped_gemm(B.GROUPED_FWD, xq, xe, wq.q_row, wq.e8_row, group_end, G, M, N, K, y, ws, stream)
    return y


def mx_moe_backward(dy: torch.Tensor, x: torch.Tensor, wq: MxExpertWeights, group_end: torch.Tensor,
                    mode: int = B.MX_RCEIL, stream=None):
    M, N = dy.shape
    K = x.shape[1]
    G = wq.q_row.shape[0]
    # dy rowwise (dgrad) and colwise (wgrad) from one read of dy.
    dyq, dye = B.alloc_mx_row(dy)
    dyqT, dyeT = B.alloc_mx_col(dy)
    B.mxfp8_quant_1x32_rowcol(dy, dyq, dye, dyqT, dyeT, mode, stream)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=dy.device)
    ws = B.alloc_grouped_workspace(B.GROUPED_DGRAD, G, M, N, K, dy.device)
    B.mxfp8_grouped_gemm(B.GROUPED_DGRAD, dyq, dye, wq.qT_col, wq.e8_col, group_end, G, M, N, K, dx, ws, stream)
    xqT, xeT = B.alloc_mx_col(x)
    B.mxfp8_quant_1x32_col(x, xqT, xeT, mode, stream)
    dW = torch.empty((G, N, K), dtype=torch.bfloat16, device=dy.device)
    ws = B.alloc_grouped_workspace(B.GROUPED_WGRAD, G, M, N, K, dy.device)
    B.mxfp8_grouped_gemm(B.GROUPED_WGRAD, dyqT, dyeT, xqT, xeT, group_end, G, M, N, K, dW, ws, stream)
    return dx, dW


# ------------------------------------------------------------------ preallocated step

class BlockwiseLinearWorkspace:
    """Every output of one Float8BlockwiseLinear forward+backward, allocated once.

    ``kernels(x, w, dy)`` lists the step's library calls in order as
    (name, callable) pairs, so a caller can time each one; ``step`` runs them.
    Inputs: x [M, K], w [N, K], dy [M, N] bf16 on the workspace's device.
    With ``weight_transpose`` the weight quantizer also writes q_W^T and dgrad
    reads that copy instead of q_W.
    """

    NAMES = ("quant_1x128_rowcol(x)", "quant_128x128(W)", "gemm_fwd", "quant_1x128_rowcol(dy)", "gemm_dgrad",
             "gemm_wgrad")

    def __init__(self, M: int, N: int, K: int, device="cuda", weight_transpose: bool = False):
        self.M, self.N, self.K = M, N, K
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)  # noqa: E731
        self.xq, self.xs = e((M, K), u8), e((K // 128, M), f32)
        self.wq, self.wqT = e((N, K), u8), (e((K, N), u8) if weight_transpose else None)
        self.ws = torch.zeros((N // 128, B.scale_ld_128x128(K)), dtype=f32, device=device)
        self.y = e((M, N), bf)
        self.dyq, self.dys = e((M, N), u8), e((N // 128, M), f32)
        self.dx = e((M, K), bf)
        self.dyqT, self.dysT = e((N, M), u8), e((M // 128, N), f32)
        self.xqT, self.xsT = e((K, M), u8), e((M // 128, K), f32)
        self.dW = e((N, K), bf)
        self.wgrad_ws = B.alloc_wgrad_workspace(M, N, K, device)  # tail split of wgrad (None if not needed)

    def kernels(self, x, w, dy, stream=None):
        return [
            ("quant_1x128_rowcol(x)",
             lambda: B.fp8bw_quant_1x128_rowcol(x, self.xq, self.xs, self.xqT, self.xsT, stream)),
            ("quant_128x128(W)", lambda: B.fp8bw_quant_128x128(w, self.wq, self.wqT, self.ws, stream)),
            ("gemm_fwd", lambda: B.fp8bw_gemm_fwd(self.xq, self.xs, self.wq, self.ws, self.y, stream)),
            ("quant_1x128_rowcol(dy)",
             lambda: B.fp8bw_quant_1x128_rowcol(dy, self.dyq, self.dys, self.dyqT, self.dysT, stream)),
            ("gemm_dgrad",
             lambda: B.fp8bw_gemm_dgrad(self.dyq, self.dys, self.wq, self.wqT, self.ws, self.dx, stream)),
            ("gemm_wgrad",
             lambda: B.fp8bw_gemm_wgrad_ws(self.dyqT, self.dysT, self.xqT, self.xsT, self.dW, self.wgrad_ws, stream)),
        ]

    def step(self, x, w, dy, stream=None):
        for _, fn in self.kernels(x, w, dy, stream):
            fn()
        return self.y, self.dx, self.dW

    def algorithmic(self):
        """Per-kernel algorithmic work: bytes moved (quantizers) or flops (GEMMs)."""
        M, N, K = self.M, self.N, self.K
        # bf16 in once; e4m3 out twice (rowwise and colwise); one fp32 per 128 each way
        rowcol = lambda r, c: r * c * 4 + 2 * 4 * r * c // 128  # noqa: E731
        return {
            "quant_1x128_rowcol(x)": ("bytes", rowcol(M, K)),
            "quant_128x128(W)": ("bytes", N * K * (3 if self.wqT is None else 4) + 4 * (N // 128) * (K // 128)),
            "gemm_fwd": ("flops", 2 * M * N * K),
            "quant_1x128_rowcol(dy)": ("bytes", rowcol(M, N)),
            "gemm_dgrad": ("flops", 2 * M * N * K),
            "gemm_wgrad": ("flops", 2 * M * N * K),
        }


class MxMoEWorkspace:
    """Every output of one MXFP8 MoE grouped linear forward+backward, allocated once.

    Inputs: x [M, K], w [G, N, K], dy [M, N] bf16 and group_end int32 [G] on
    the workspace's device.  ``kernels`` lists the step's six library calls:
    each of x, W and dy is read once for both its MX quantizations.
    """

    def __init__(self, M: int, N: int, K: int, G: int, device="cuda", mode: int = B.MX_RCEIL):
        self.M, self.N, self.K, self.G, self.mode = M, N, K, G, mode
        u8, bf = torch.uint8, torch.bfloat16
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)  # noqa: E731
        self.xq, self.xe = e((M, K), u8), e((M, K // 32), u8)
        self.wq, self.we = e((G * N, K), u8), e((G * N, K // 32), u8)
        self.wqT, self.weT = e((G, K, N), u8), e((G, K, N // 32), u8)
        self.y = e((M, N), bf)
        self.dyq, self.dye = e((M, N), u8), e((M, N // 32), u8)
        self.dx = e((M, K), bf)
        self.dyqT, self.dyeT = e((N, M), u8), e((N, M // 32), u8)
        self.xqT, self.xeT = e((K, M), u8), e((K, M // 32), u8)
        self.dW = e((G, N, K), bf)
        self.ws = e((max(B.mxfp8_grouped_gemm_workspace_bytes(k, G, M, N, K) for k in range(3)),), u8)

    def kernels(self, x, w, dy, group_end, stream=None):
        M, N, K, G, md = self.M, self.N, self.K, self.G, self.mode
        return [
            ("mx_quant_1x32_rowcol(x)", lambda: B.mxfp8_quant_1x32_rowcol(x, self.xq, self.xe, self.xqT, self.xeT,
                                                                          md, stream)),
            ("mx_quant_1x32_rowcol(W)", lambda: B.mxfp8_quant_1x32_rowcol(w, self.wq, self.we, self.wqT, self.weT,
                                                                          md, stream)),
            ("mx_grouped_fwd", lambda: B.mxfp8_grouped_gemm(B.GROUPED_FWD, self.xq, self.xe, self.wq, self.we,
                                                            group_end, G, M, N, K, self.y, self.ws, stream)),
            ("mx_quant_1x32_rowcol(dy)", lambda: B.mxfp8_quant_1x32_rowcol(dy, self.dyq, self.dye, self.dyqT,
                                                                           self.dyeT, md, stream)),
            ("mx_grouped_dgrad", lambda: B.mxfp8_grouped_gemm(B.GROUPED_DGRAD, self.dyq, self.dye, self.wqT,
                                                              self.weT, group_end, G, M, N, K, self.dx, self.ws, stream)),
            ("mx_grouped_wgrad", lambda: B.mxfp8_grouped_gemm(B.GROUPED_WGRAD, self.dyqT, self.dyeT, self.xqT,
                                                              self.xeT, group_end, G, M, N, K, self.dW, self.ws, stream)),
        ]

    def step(self, x, w, dy, group_end, stream=None):
        for _, fn in self.kernels(x, w, dy, group_end, stream):
            fn()
        return self.y, self.dx, self.dW

    def algorithmic(self):
        M, N, K, G = self.M, self.N, self.K, self.G
        # bf16 in once; e4m3 out twice (rowwise and colwise); one E8M0 byte per 32 each way
        mx2 = lambda r, c: r * c * 4 + 2 * (r * c // 32)  # noqa: E731
        return {
            "mx_quant_1x32_rowcol(x)": ("bytes", mx2(M, K)),
            "mx_quant_1x32_rowcol(W)": ("bytes", mx2(G * N, K)),
            "mx_grouped_fwd": ("flops", 2 * M * N * K),
            "mx_quant_1x32_rowcol(dy)": ("bytes", mx2(M, N)),
            "mx_grouped_dgrad": ("flops", 2 * M * N * K),
            "mx_grouped_wgrad": ("flops", 2 * M * N * K),
        }


class PipelinedLinearSteps:
    """Forward+backward steps of a blockwise-FP8 linear fed from and drained to
    pinned host memory, with the copies of neighbouring steps overlapping the
    kernels.

    Step i uses device buffer set i % 2: its inputs are copied host->device on
    an upload stream, the six library calls of ``BlockwiseLinearWorkspace.step``
    run on a compute stream once they have landed, and y, dx, dW are copied
    device->host on a download stream once computed.  Events order each use of
    a buffer set after the previous step that used it (upload after that
    step's kernels read the inputs, kernels after that step's download read
    the outputs), so step i + 1's upload and step i - 1's download run while
    step i computes.
    """

    def __init__(self, M: int, N: int, K: int, device="cuda"):
        bf = torch.bfloat16
        e = lambda shape: torch.empty(shape, dtype=bf, device=device)  # noqa: E731
        self.inputs = [(e((M, K)), e((N, K)), e((M, N))) for _ in range(2)]
        self.ws = [BlockwiseLinearWorkspace(M, N, K, device=device) for _ in range(2)]
        self.up, self.comp, self.down = (torch.cuda.Stream(device=device) for _ in range(3))
        mk = lambda: [torch.cuda.Event() for _ in range(2)]  # noqa: E731
        self.uploaded, self.computed, self.downloaded = mk(), mk(), mk()
        self.i = 0

    def step(self, x_h, w_h, dy_h, y_h, dx_h, dW_h) -> None:
        """Enqueues one step: host inputs x_h, w_h, dy_h (pinned bf16) in,
        host outputs y_h, dx_h, dW_h (pinned bf16) out.  Returns at once;
        ``synchronize`` waits for every enqueued step."""
        for name, t in (("x_h", x_h), ("w_h", w_h), ("dy_h", dy_h), ("y_h", y_h), ("dx_h", dx_h), ("dW_h", dW_h)):
            if t.device.type != "cpu" or not t.is_pinned():
                raise ValueError(f"{name} must be a pinned host tensor")
        s = self.i % 2
        x, w, dy = self.inputs[s]
        ws = self.ws[s]
        if self.i >= 2:
            self.up.wait_event(self.computed[s])
            self.comp.wait_event(self.downloaded[s])
        with torch.cuda.stream(self.up):
            x.copy_(x_h, non_blocking=True)
            w.copy_(w_h, non_blocking=True)
            dy.copy_(dy_h, non_blocking=True)
            self.uploaded[s].record(self.up)
        self.comp.wait_event(self.uploaded[s])
        ws.step(x, w, dy, stream=self.comp)
        self.computed[s].record(self.comp)
        self.down.wait_event(self.computed[s])
        with torch.cuda.stream(self.down):
            y_h.copy_(ws.y, non_blocking=True)
            dx_h.copy_(ws.dx, non_blocking=True)
            dW_h.copy_(ws.dW, non_blocking=True)
            self.downloaded[s].record(self.down)
        self.i += 1

    def synchronize(self) -> None:
        for st in (self.up, self.comp, self.down):
            st.synchronize()


class ToyFFNStep:
    """Forward+backward of the toy FFN of PR #4295 ("add FSDP and TP tests for
    Float8BlockwiseLinear", Summary: the ToyModel's w1, w2 and out_proj under
    the standard FFN plan), out = out_proj(silu(w1 x) * (w2 x)), with every
    GEMM a blockwise-FP8 library call and every output preallocated.

    Inputs: x [M, dim], w1, w2 [hidden, dim], wo [dim, hidden], dy [M, dim]
    bf16.  x is quantized once (rowwise and colwise in one pass) for both
    up-projections.  The silu * mul activation and its derivative are the
    model's own elementwise code (not part of the library), run as the bf16
    torch ops that autograd runs for ``silu(h1) * h2``: silu(h1) and the
    product are each rounded to bf16; backward, g = da * h2, dh1 =
    silu_backward(g, h1) and dh2 = da * silu(h1), each rounded to bf16.
    ``kernels`` lists the step's
    calls in order as (name, callable) pairs for per-call timing; names of
    library GEMMs start with "gemm".
    """

    NAMES = ("quant_1x128_rowcol(x)", "quant_128x128(w1)", "quant_128x128(w2)", "quant_128x128(out_proj)",
             "gemm_fwd(w1)", "gemm_fwd(w2)", "act silu*mul (torch)", "quant_1x128_rowcol(a)", "gemm_fwd(out_proj)",
             "quant_1x128_rowcol(dy)", "gemm_dgrad(out_proj)", "gemm_wgrad(out_proj)", "act grad (torch)",
             "quant_1x128_rowcol(dh1)", "quant_1x128_rowcol(dh2)", "gemm_dgrad(w1)", "gemm_wgrad(w1)",
             "gemm_dgrad(w2)", "gemm_wgrad(w2)", "dx sum (torch)")

    def __init__(self, M: int, dim: int, hidden: int, device="cuda"):
        self.M, self.dim, self.hidden = M, dim, hidden
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)  # noqa: E731

        def act(R, C):
            return {"q": e((R, C), u8), "s": e((C // 128, R), f32), "qT": e((C, R), u8), "sT": e((R // 128, C), f32)}

        def wt(R, C):
            return QuantizedWeight(e((R, C), u8), None,
                                   torch.zeros((R // 128, B.scale_ld_128x128(C)), dtype=f32, device=device))

        self.xa, self.aa, self.dya, self.dh1a, self.dh2a = act(M, dim), act(M, hidden), act(M, dim), \
            act(M, hidden), act(M, hidden)
        self.w1q, self.w2q, self.woq = wt(hidden, dim), wt(hidden, dim), wt(dim, hidden)
        self.h1, self.h2, self.a = e((M, hidden), bf), e((M, hidden), bf), e((M, hidden), bf)
        self.s1, self.g = e((M, hidden), bf), e((M, hidden), bf)  # silu(h1) (kept for backward), da * h2
        self.out, self.da, self.dh1, self.dh2 = e((M, dim), bf), e((M, hidden), bf), e((M, hidden), bf), \
            e((M, hidden), bf)
        self.dx1, self.dx2, self.dx = e((M, dim), bf), e((M, dim), bf), e((M, dim), bf)
        self.d_w1, self.d_w2, self.d_wo = e((hidden, dim), bf), e((hidden, dim), bf), e((dim, hidden), bf)
        # one workspace for the three wgrads (they run one after another on one stream)
        sizes = [B.fp8bw_gemm_wgrad_workspace_bytes(M, dim, hidden), B.fp8bw_gemm_wgrad_workspace_bytes(M, hidden, dim)]
        self.wgrad_ws = e((max(sizes),), u8) if max(sizes) else None

    @staticmethod
    def _rowcol(src, a, stream):
        return lambda: B.fp8bw_quant_1x128_rowcol(src, a["q"], a["s"], a["qT"], a["sT"], stream)

    def _act(self):
        torch.ops.aten.silu.out(self.h1, out=self.s1)
        torch.mul(self.s1, self.h2, out=self.a)

    def _act_grad(self):
        torch.mul(self.da, self.h2, out=self.g)
        torch.ops.aten.silu_backward.grad_input(self.g, self.h1, grad_input=self.dh1)
        torch.mul(self.da, self.s1, out=self.dh2)

    def kernels(self, x, w1, w2, wo, dy, stream=None):
        xa, aa, dya, d1, d2 = self.xa, self.aa, self.dya, self.dh1a, self.dh2a
        q1, q2, qo = self.w1q, self.w2q, self.woq
        return [
            ("quant_1x128_rowcol(x)", self._rowcol(x, xa, stream)),
            ("quant_128x128(w1)", lambda: B.fp8bw_quant_128x128(w1, q1.q, q1.qT, q1.s, stream)),
            ("quant_128x128(w2)", lambda: B.fp8bw_quant_128x128(w2, q2.q, q2.qT, q2.s, stream)),
            ("quant_128x128(out_proj)", lambda: B.fp8bw_quant_128x128(wo, qo.q, qo.qT, qo.s, stream)),
            ("gemm_fwd(w1)", lambda: B.fp8bw_gemm_fwd(xa["q"], xa["s"], q1.q, q1.s, self.h1, stream)),
            ("gemm_fwd(w2)", lambda: B.fp8bw_gemm_fwd(xa["q"], xa["s"], q2.q, q2.s, self.h2, stream)),
            ("act silu*mul (torch)", self._act),
            ("quant_1x128_rowcol(a)", self._rowcol(self.a, aa, stream)),
            ("gemm_fwd(out_proj)", lambda: B.fp8bw_gemm_fwd(aa["q"], aa["s"], qo.q, qo.s, self.out, stream)),
            ("quant_1x128_rowcol(dy)", self._rowcol(dy, dya, stream)),
            ("gemm_dgrad(out_proj)",
             lambda: B.fp8bw_gemm_dgrad(dya["q"], dya["s"], qo.q, qo.qT, qo.s, self.da, stream)),
            ("gemm_wgrad(out_proj)",
             lambda: B.fp8bw_gemm_wgrad_ws(dya["qT"], dya["sT"], aa["qT"], aa["sT"], self.d_wo, self.wgrad_ws, stream)),
            ("act grad (torch)", self._act_grad),
            ("quant_1x128_rowcol(dh1)", self._rowcol(self.dh1, d1, stream)),
            ("quant_1x128_rowcol(dh2)", self._rowcol(self.dh2, d2, stream)),
            ("gemm_dgrad(w1)", lambda: B.fp8bw_gemm_dgrad(d1["q"], d1["s"], q1.q, q1.qT, q1.s, self.dx1, stream)),
            ("gemm_wgrad(w1)",
             lambda: B.fp8bw_gemm_wgrad_ws(d1["qT"], d1["sT"], xa["qT"], xa["sT"], self.d_w1, self.wgrad_ws, stream)),
            ("gemm_dgrad(w2)", lambda: B.fp8bw_gemm_dgrad(d2["q"], d2["s"], q2.q, q2.qT, q2.s, self.dx2, stream)),
            ("gemm_wgrad(w2)",
             lambda: B.fp8bw_gemm_wgrad_ws(d2["qT"], d2["sT"], xa["qT"], xa["sT"], self.d_w2, self.wgrad_ws, stream)),
            ("dx sum (torch)", lambda: torch.add(self.dx1, self.dx2, out=self.dx)),
        ]

    def step(self, x, w1, w2, wo, dy, stream=None):
        for _, fn in self.kernels(x, w1, w2, wo, dy, stream):
            fn()
        return {"out": self.out, "dx": self.dx, "d_w1": self.d_w1, "d_w2": self.d_w2, "d_out_proj": self.d_wo}

    def algorithmic(self):
        """Per-call algorithmic work: flops (GEMMs), bytes (quantizers), None (model's torch ops)."""
        M, D, H = self.M, self.dim, self.hidden
        rowcol = lambda r, c: r * c * 4 + 2 * 4 * r * c // 128  # noqa: E731
        w128 = lambda r, c: r * c * 3 + 4 * (r // 128) * (c // 128)  # noqa: E731
        g = 2 * M * D * H
        out = {}
        for n in self.NAMES:
            if n.startswith("gemm"):
                out[n] = ("flops", g)
            elif n.startswith("quant_128x128"):
                out[n] = ("bytes", w128(D, H))
            elif n.startswith("quant_1x128_rowcol"):
                out[n] = ("bytes", rowcol(M, D if n.endswith("(x)") or n.endswith("(dy)") else H))
            else:
                out[n] = (None, 0)
        return out
