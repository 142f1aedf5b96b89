"""mxfp8_grouped_gemm_noalloc: the grouped GEMM for callers that cannot allocate
device memory (code that only holds pointers handed out by a framework that
owns every allocation, or a loop whose device footprint is fixed up front).
It uses the library's fixed scratch array instead of a caller workspace; this
test checks, through the C ABI, that two calls in a row give what the
workspace entry point gives for every kind.  The file is named to be collected
last, so a failure here leaves every other test already run."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
from mxfp8_precision_gemms_fp8bw_gb300 import inputs

pytestmark = pytest.mark.gpu


def _operands(kind, x, w, dy):
    """Quantized operands of one kind, from the library's own quantizers."""
    G, N, K = w.shape
    M = x.shape[0]
    if kind == B.GROUPED_FWD:
        a, ae = B.alloc_mx_row(x)
        B.mxfp8_quant_1x32_row(x, a, ae)
        b, be = B.alloc_mx_row(w.view(G * N, K))
        B.mxfp8_quant_1x32_row(w.view(G * N, K), b, be)
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    elif kind == B.GROUPED_DGRAD:
        a, ae = B.alloc_mx_row(dy)
        B.mxfp8_quant_1x32_row(dy, a, ae)
        b, be = B.alloc_mx_3d_col(w)
        B.mxfp8_quant_3d_col(w, b, be)
        out = torch.empty((M, K), dtype=torch.bfloat16, device=x.device)
    else:
        a, ae = B.alloc_mx_col(dy)
        B.mxfp8_quant_1x32_col(dy, a, ae)
        b, be = B.alloc_mx_col(x)
        B.mxfp8_quant_1x32_col(x, b, be)
        out = torch.empty((G, N, K), dtype=torch.bfloat16, device=x.device)
    return a, ae, b, be, out


def _oracle_error(kind, a, ae, b, be, group_end, G, M, N, K, got):
    """Largest per-element normalized error of a grouped GEMM output against
    the oracle on the same quantized operands (group by group)."""
    u = lambda t: t.cpu().numpy()  # noqa: E731
    ref = oracle.mx_grouped_gemm(kind, u(a), u(ae), u(b), u(be), group_end, G, M, N, K)
    got = got.float().cpu().numpy()
    if kind == B.GROUPED_FWD:
        ad, bd = oracle.mx_dequant_row(u(a), u(ae)), oracle.mx_dequant_row(u(b), u(be)).reshape(G, N, K)
    elif kind == B.GROUPED_DGRAD:
        ad, bd = oracle.mx_dequant_row(u(a), u(ae)), oracle.mx_dequant_row(u(b).reshape(G * K, N),
                                                                             u(be).reshape(G * K, N // 32)).reshape(G, K, N)
    else:
        ad, bd = oracle.mx_dequant_row(u(a), u(ae)), oracle.mx_dequant_row(u(b), u(be))
    err = 0.0
    for g, (lo, hi) in enumerate(zip(oracle.group_starts(group_end), group_end)):
        if kind == B.GROUPED_WGRAD:
            e = oracle.normalized_gemm_error(got[g], ref[g], oracle.row_norms(ad[:, lo:hi]), oracle.row_norms(bd[:, lo:hi]))
        elif hi > lo:
            e = oracle.normalized_gemm_error(got[lo:hi], ref[lo:hi], oracle.row_norms(ad[lo:hi]), oracle.row_norms(bd[g]))
        else:
            continue
        err = max(err, float(e.max()))
    return err


def test_noalloc_matches_workspace_entry_point_twice():
    B.lib(build_if_missing=True)
    rng = np.random.default_rng(21)
    M, K, N, G = 768, 512, 512, 4
    group_end = np.array([160, 160, 544, 768], np.int32)      # an empty group, 32-aligned boundaries
    x = inputs.normal_bf16(rng, (M, K), 1.0).cuda()
    w = inputs.normal_bf16(rng, (G, N, K), 0.02).cuda()
    dy = inputs.normal_bf16(rng, (M, N), 1e-3).cuda()
    ge = torch.from_numpy(group_end).cuda()
    for kind in (B.GROUPED_FWD, B.GROUPED_DGRAD, B.GROUPED_WGRAD):
        a, ae, b, be, ref = _operands(kind, x, w, dy)
        ws = B.alloc_grouped_workspace(kind, G, M, N, K, x.device)
        B.mxfp8_grouped_gemm(kind, a, ae, b, be, ge, G, M, N, K, ref, ws)
        B.fp8bw_sync_status()
        # the workspace entry point against the oracle
        assert _oracle_error(kind, a, ae, b, be, group_end, G, M, N, K, ref) <= oracle.GEMM_TOL, kind
        # Two calls in a row on the shared array, the first after another
        # kind's calls left different packed scales in it: both must equal the
        # workspace call bit for bit (same kernels, same packed scales), so a
        # stale or partly rewritten scratch word would show.
        for _ in range(2):
            out = torch.full_like(ref, float("nan"))
            B.mxfp8_grouped_gemm_noalloc(kind, a, ae, b, be, ge, G, M, N, K, out)
            B.fp8bw_sync_status()
            assert torch.equal(out, ref), kind


def test_noalloc_rejects_dims_beyond_the_fixed_scratch():
    B.lib(build_if_missing=True)
    need = B.mxfp8_grouped_gemm_workspace_bytes(B.GROUPED_DGRAD, 8, 16384, 16384, 16384)
    assert need > B.NOALLOC_SCRATCH_BYTES
    t = torch.empty(16, dtype=torch.uint8, device="cuda")
    ge = torch.zeros(8, dtype=torch.int32, device="cuda")
    out = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.Fp8bwError) as e:
        B.mxfp8_grouped_gemm_noalloc(B.GROUPED_DGRAD, t, t, t, t, ge, 8, 16384, 16384, 16384, out)
    assert e.value.code == B.ERR_SHAPE and "scratch" in str(e.value)
