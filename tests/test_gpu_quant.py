"""GPU parity of the quantizers: bit-exact e4m3 bytes and scale bits vs the oracle.

Covers several tiles with ragged edges (MX), the edge cases of
``gpu_util.adversarial_bf16``, both MX exponent modes, every finite bf16
value as a block max (1x128 and 1x32, rowwise and colwise), and the full-size dense
linear workload (x[16384, 5120], W[8192, 5120], dy[16384, 8192]) and the
full-size MXFP8 MoE tensors (x[16384, 5120], dy[16384, 8192] rowwise and
colwise, the expert weights W[8, 8192, 5120] rowwise and 3D colwise),
compared byte for byte in row chunks.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import adversarial_bf16, bits, dense_inputs, f32, lib, oracle_map, transpose_adversarial, u8
from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
from mxfp8_precision_gemms_fp8bw_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()


def run_row(x):
    xd = x.cuda()
    q, s = B.alloc_quant_1x128_row(xd)
    B.fp8bw_quant_1x128_row(xd, q, s)
    B.fp8bw_sync_status()
    return u8(q), s.cpu().numpy()


def run_col(x):
    xd = x.cuda()
    qT, s = B.alloc_quant_1x128_col(xd)
    B.fp8bw_quant_1x128_col(xd, qT, s)
    B.fp8bw_sync_status()
    return u8(qT), s.cpu().numpy()


def run_128(x, with_t=True):
    xd = x.cuda()
    q, qT, s = B.alloc_quant_128x128(xd, with_t)
    B.fp8bw_quant_128x128(xd, q, qT, s)
    B.fp8bw_sync_status()
    return u8(q), (u8(qT) if with_t else None), s.cpu().numpy()


@pytest.mark.parametrize("R,C,seed", [(128, 128, 0), (256, 512, 1), (384, 640, 2), (1152, 896, 3)])
def test_1x128_row_bit_exact(R, C, seed):
    x = adversarial_bf16(R, C, seed)
    q, s = run_row(x)
    qo, so = oracle.quant_1x128_row(f32(x))
    assert np.array_equal(q, qo)
    assert np.array_equal(bits(s), bits(so))


@pytest.mark.parametrize("R,C,seed", [(128, 128, 4), (256, 512, 5), (640, 384, 6), (1024, 1152, 7)])
def test_1x128_col_bit_exact(R, C, seed):
    x = transpose_adversarial(R, C, seed)
    qT, s = run_col(x)
    qo, so = oracle.quant_1x128_col(f32(x))
    assert np.array_equal(qT, qo)
    assert np.array_equal(bits(s), bits(so))


@pytest.mark.parametrize("R,C,seed", [(128, 128, 11), (256, 512, 12), (640, 384, 13), (1152, 896, 14)])
def test_1x128_rowcol_bit_exact(R, C, seed):
    # one read of x, both outputs: identical to the separate row and col quantizers
    x = adversarial_bf16(R, C, seed) if seed % 2 else transpose_adversarial(R, C, seed)
    xd = x.cuda()
    q, s = B.alloc_quant_1x128_row(xd)
    qT, sT = B.alloc_quant_1x128_col(xd)
    B.fp8bw_quant_1x128_rowcol(xd, q, s, qT, sT)
    B.fp8bw_sync_status()
    qo, so = oracle.quant_1x128_row(f32(x))
    qTo, sTo = oracle.quant_1x128_col(f32(x))
    assert np.array_equal(u8(q), qo) and np.array_equal(bits(s), bits(so))
    assert np.array_equal(u8(qT), qTo) and np.array_equal(bits(sT), bits(sTo))


@pytest.mark.parametrize("R,C,seed", [(128, 128, 8), (384, 640, 9), (512, 384, 10)])
def test_128x128_bit_exact(R, C, seed):
    x = adversarial_bf16(R, C, seed)
    q, qT, s = run_128(x)
    qo, qTo, so = oracle.quant_128x128(f32(x))
    assert np.array_equal(q, qo)
    assert np.array_equal(qT, qTo)
    ld = B.scale_ld_128x128(C)
    assert s.shape == (R // 128, ld)
    assert np.array_equal(bits(s[:, :C // 128]), bits(so))
    assert np.all(s[:, C // 128:] == 0)         # padding untouched (allocated zeroed)
    q2, _, s2 = run_128(x, with_t=False)        # qT is optional
    assert np.array_equal(q2, qo) and np.array_equal(bits(s2[:, :C // 128]), bits(so))


def test_signed_zero_and_ties_on_device():
    # amax = 448 -> s = 1: 10.5 -> 0x52, 11.5 -> 0x54, -0.0 -> 0x80, 3*2^-10 -> 0x02.
    row = np.zeros(128, np.float32)
    row[:5] = [448.0, 10.5, 11.5, -0.0, 3 * 2.0 ** -10]
    x = torch.from_numpy(np.tile(row, (128, 1))).to(torch.bfloat16)
    q, s = run_row(x)
    assert list(q[0, :5]) == [0x7E, 0x52, 0x54, 0x80, 0x02]
    assert np.all(s == 1.0)


def test_1x128_every_bf16_block_max():
    # The blockwise scale and the division over every finite bf16 block max
    # (zero takes the 1e-12 floor), rowwise and -- on the transpose --
    # colwise, through the separate and the fused kernels.
    x = _every_bf16_block_max(50, width=128)
    xT = x.t().contiguous()  # [128, 32640]
    qo, so = oracle.quant_1x128_row(f32(x))
    qTo, sTo = oracle.quant_1x128_col(f32(xT))
    assert np.array_equal(qTo, qo) and np.array_equal(bits(sTo).reshape(-1), bits(so).reshape(-1))
    q, s = run_row(x)
    assert np.array_equal(q, qo) and np.array_equal(bits(s), bits(so))
    qT, sT = run_col(xT)
    assert np.array_equal(qT, qTo) and np.array_equal(bits(sT), bits(sTo))
    xd = x.cuda()
    q, s = B.alloc_quant_1x128_row(xd)
    qT, sT = B.alloc_quant_1x128_col(xd)
    B.fp8bw_quant_1x128_rowcol(xd, q, s, qT, sT)
    B.fp8bw_sync_status()
    assert np.array_equal(u8(q), qo) and np.array_equal(bits(s.cpu().numpy()), bits(so))


# ---------------------------------------------------------------- MXFP8

@pytest.mark.parametrize("mode", [B.MX_RCEIL, B.MX_FLOOR])
@pytest.mark.parametrize("R,C,seed", [(32, 32, 0), (96, 160, 1), (257, 544, 2), (512, 1024, 3)])
def test_mx_row_bit_exact(mode, R, C, seed):
    x = adversarial_bf16(R, C, seed, block=32)
    xd = x.cuda()
    q, e8 = B.alloc_mx_row(xd)
    B.mxfp8_quant_1x32_row(xd, q, e8, mode)
    B.fp8bw_sync_status()
    qo, eo = oracle.mx_quant_1x32_row(f32(x), mode)
    assert np.array_equal(u8(q), qo)
    assert np.array_equal(u8(e8), eo)


@pytest.mark.parametrize("mode", [B.MX_RCEIL, B.MX_FLOOR])
@pytest.mark.parametrize("R,C,seed", [(32, 8, 0), (96, 136, 1), (160, 256, 2), (544, 520, 3)])
def test_mx_col_bit_exact(mode, R, C, seed):
    x = transpose_adversarial(R, C, seed, block=32)
    xd = x.cuda()
    qT, e8 = B.alloc_mx_col(xd)
    B.mxfp8_quant_1x32_col(xd, qT, e8, mode)
    B.fp8bw_sync_status()
    qo, eo = oracle.mx_quant_1x32_col(f32(x), mode)
    assert np.array_equal(u8(qT), qo)
    assert np.array_equal(u8(e8), eo)


@pytest.mark.parametrize("mode", [B.MX_RCEIL, B.MX_FLOOR])
def test_mx_3d_col_bit_exact(mode):
    G, N, K = 3, 160, 264
    w = torch.stack([transpose_adversarial(N, K, 10 + g, block=32) for g in range(G)])
    wd = w.cuda()
    qT, e8 = B.alloc_mx_3d_col(wd)
    B.mxfp8_quant_3d_col(wd, qT, e8, mode)
    B.fp8bw_sync_status()
    qo, eo = oracle.mx_quant_3d_col(f32(w), mode)
    assert np.array_equal(u8(qT), qo)
    assert np.array_equal(u8(e8), eo)


def _mx_rowcol(x, mode):
    """Both MX quantizations of x ([R, C] or [G, R, C]) from the fused kernel."""
    xd = x.cuda()
    G, R, C = (1, *x.shape) if x.dim() == 2 else x.shape
    q = torch.empty((G * R, C), dtype=torch.uint8, device="cuda")
    e8 = torch.empty((G * R, C // 32), dtype=torch.uint8, device="cuda")
    qT = torch.empty((G, C, R), dtype=torch.uint8, device="cuda")
    e8T = torch.empty((G, C, R // 32), dtype=torch.uint8, device="cuda")
    B.mxfp8_quant_1x32_rowcol(xd, q, e8, qT, e8T, mode)
    B.fp8bw_sync_status()
    return u8(q), u8(e8), u8(qT), u8(e8T)


@pytest.mark.parametrize("mode", [B.MX_RCEIL, B.MX_FLOOR])
@pytest.mark.parametrize("R,C,seed", [(32, 32, 20), (96, 160, 21), (288, 544, 22), (544, 256, 23)])
def test_mx_rowcol_bit_exact(mode, R, C, seed):
    # The fused kernel against both oracle quantizers, on blocks adversarial
    # along the rows (rowwise pass) and along the columns (colwise pass).
    for x in (adversarial_bf16(R, C, seed, block=32), transpose_adversarial(R, C, seed, block=32)):
        q, e8, qT, e8T = _mx_rowcol(x, mode)
        qo, eo = oracle.mx_quant_1x32_row(f32(x), mode)
        qTo, eTo = oracle.mx_quant_1x32_col(f32(x), mode)
        assert np.array_equal(q, qo) and np.array_equal(e8, eo)
        assert np.array_equal(qT[0], qTo) and np.array_equal(e8T[0], eTo)


@pytest.mark.parametrize("mode", [B.MX_RCEIL, B.MX_FLOOR])
def test_mx_rowcol_3d_bit_exact(mode):
    # Stacked expert weights [G, N, K]: rowwise along K over [G*N, K], and the
    # 3D colwise (32 along N per expert, written [G, K, N]).
    G, N, K = 3, 160, 288
    w = torch.stack([transpose_adversarial(N, K, 30 + g, block=32) for g in range(G)])
    q, e8, qT, e8T = _mx_rowcol(w, mode)
    qo, eo = oracle.mx_quant_1x32_row(f32(w).reshape(G * N, K), mode)
    qTo, eTo = oracle.mx_quant_3d_col(f32(w), mode)
    assert np.array_equal(q, qo) and np.array_equal(e8, eo)
    assert np.array_equal(qT, qTo) and np.array_equal(e8T, eTo)


def _every_bf16_block_max(seed, width=32):
    """[32640, width] bf16: row i's block max is the finite bf16 magnitude
    with bits i (0x0000 .. 0x7F7F: zero, every subnormal and every normal),
    the other elements bf16(max * u) with u uniform in [-1, 1]."""
    amax = (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    u = np.random.default_rng(seed).uniform(-1.0, 1.0, size=(amax.size, width)).astype(np.float32)
    x = amax[:, None] * u
    x[:, 0] = amax
    xb = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(np.abs(f32(xb)).max(axis=1), amax)
    return xb


@pytest.mark.parametrize("mode", [B.MX_RCEIL, B.MX_FLOOR])
def test_mx_every_bf16_block_max(mode):
    # The E8M0 exponent and 2^-E over every finite bf16 block max, through
    # the rowwise and colwise MX kernels and the fused one, against the
    # oracle's rule (reading 9, itself pinned by brute force in
    # test_oracle_mx.py).
    x = _every_bf16_block_max(40 + mode)
    xT = x.t().contiguous()  # [32, 32640]: the same blocks down the columns
    qo, eo = oracle.mx_quant_1x32_row(f32(x), mode)
    qTo, eTo = oracle.mx_quant_1x32_col(f32(xT), mode)
    assert np.array_equal(qTo, qo) and np.array_equal(eTo.reshape(-1), eo.reshape(-1))

    xd = x.cuda()
    q, e8 = B.alloc_mx_row(xd)
    B.mxfp8_quant_1x32_row(xd, q, e8, mode)
    B.fp8bw_sync_status()
    assert np.array_equal(u8(q), qo) and np.array_equal(u8(e8), eo)

    xTd = xT.cuda()
    qT, e8T = B.alloc_mx_col(xTd)
    B.mxfp8_quant_1x32_col(xTd, qT, e8T, mode)
    B.fp8bw_sync_status()
    assert np.array_equal(u8(qT), qTo) and np.array_equal(u8(e8T), eTo)

    q, e8, qT, e8T = _mx_rowcol(x, mode)
    assert np.array_equal(q, qo) and np.array_equal(e8, eo)
    q, e8, qT, e8T = _mx_rowcol(xT, mode)
    assert np.array_equal(qT[0], qTo) and np.array_equal(e8T[0], eTo)


# ---------------------------------------------------------------- full size

@pytest.fixture(scope="module")
def dense():
    return dense_inputs()


def _chunks(R, step):
    for r0 in range(0, R, step):
        yield r0, min(R, r0 + step)


def test_full_size_dense_row_and_col_quant(dense):
    for t in (dense.x, dense.dy):
        td = t.cuda()
        q, s = B.alloc_quant_1x128_row(td)
        B.fp8bw_quant_1x128_row(td, q, s)
        qT, sT = B.alloc_quant_1x128_col(td)
        B.fp8bw_quant_1x128_col(td, qT, sT)
        q2, s2 = B.alloc_quant_1x128_row(td)
        qT2, sT2 = B.alloc_quant_1x128_col(td)
        B.fp8bw_quant_1x128_rowcol(td, q2, s2, qT2, sT2)
        B.fp8bw_sync_status()
        assert torch.equal(q, q2) and torch.equal(s, s2) and torch.equal(qT, qT2) and torch.equal(sT, sT2)
        q, s, qT, sT = u8(q), s.cpu().numpy(), u8(qT), sT.cpu().numpy()
        tf = f32(t)
        for r0, r1 in _chunks(tf.shape[0], 2048):
            qo, so = oracle.quant_1x128_row(np.ascontiguousarray(tf[r0:r1]))
            assert np.array_equal(q[r0:r1], qo)
            assert np.array_equal(bits(s[:, r0:r1]), bits(so))
            qTo, sTo = oracle.quant_1x128_col(np.ascontiguousarray(tf[r0:r1]))
            assert np.array_equal(qT[:, r0:r1], qTo)
            assert np.array_equal(bits(sT[r0 // 128:r1 // 128]), bits(sTo))


def test_full_size_dense_weight_quant(dense):
    # Both kernels: the staged one (with q^T) and the register-staged one
    # that runs when no q^T is asked for (the linear layer's case).
    q, qT, s = run_128(dense.w)
    q2, _, s2 = run_128(dense.w, with_t=False)
    wf = f32(dense.w)
    for r0, r1 in _chunks(wf.shape[0], 2048):
        qo, qTo, so = oracle.quant_128x128(np.ascontiguousarray(wf[r0:r1]))
        assert np.array_equal(q[r0:r1], qo)
        assert np.array_equal(qT[:, r0:r1], qTo)
        assert np.array_equal(bits(s[r0 // 128:r1 // 128, :so.shape[1]]), bits(so))
        assert np.array_equal(q2[r0:r1], qo)
        assert np.array_equal(bits(s2[r0 // 128:r1 // 128, :so.shape[1]]), bits(so))


@pytest.fixture(scope="module")
def moe_tensors():
    return inputs.moe()


def _mx_gpu(kind, t):
    """One MX quantization of the bf16 tensor t on the GPU: kind row, col or 3d."""
    td = t.cuda()
    if kind == "row":
        q, e = B.alloc_mx_row(td)
        B.mxfp8_quant_1x32_row(td, q, e)
    elif kind == "col":
        q, e = B.alloc_mx_col(td)
        B.mxfp8_quant_1x32_col(td, q, e)
    else:
        q, e = B.alloc_mx_3d_col(td)
        B.mxfp8_quant_3d_col(td, q, e)
    B.fp8bw_sync_status()
    return u8(q), u8(e)


@pytest.mark.parametrize("name", ["x", "dy", "w"])
def test_full_size_moe_mx_quant_bit_exact(moe_tensors, name):
    # Every byte of the full-size MoE tensors' MX quantizations against the
    # oracle: rowwise (1x32 along the last dim) for x, dy and W viewed as
    # [G*N, K]; colwise (32 rows, written transposed) for x and dy; 3D colwise
    # (32 along N per expert, written [G, K, N]) for W.  Both sides in RCEIL.
    # The fused row + column kernel (the MoE step's path) is checked against
    # the same oracle bytes.
    t = getattr(moe_tensors, name)
    R2 = t.reshape(-1, t.shape[-1])
    q, e = _mx_gpu("row", R2)
    fq, fe, fqT, feT = _mx_rowcol(t, B.MX_RCEIL)
    host = f32(R2)
    chunks = [(np.ascontiguousarray(host[r0:r1]),) for r0, r1 in _chunks(host.shape[0], 2048)]
    for (r0, r1), (qo, eo) in zip(_chunks(host.shape[0], 2048), oracle_map("mx_quant_1x32_row", chunks)):
        assert np.array_equal(q[r0:r1], qo), (name, "row", r0)
        assert np.array_equal(e[r0:r1], eo), (name, "row e8", r0)
        assert np.array_equal(fq[r0:r1], qo), (name, "fused row", r0)
        assert np.array_equal(fe[r0:r1], eo), (name, "fused row e8", r0)
    if name != "w":
        qT, eT = _mx_gpu("col", t)
        for (r0, r1), (qo, eo) in zip(_chunks(host.shape[0], 2048), oracle_map("mx_quant_1x32_col", chunks)):
            assert np.array_equal(qT[:, r0:r1], qo), (name, "col", r0)
            assert np.array_equal(eT[:, r0 // 32:r1 // 32], eo), (name, "col e8", r0)
            assert np.array_equal(fqT[0][:, r0:r1], qo), (name, "fused col", r0)
            assert np.array_equal(feT[0][:, r0 // 32:r1 // 32], eo), (name, "fused col e8", r0)
    else:
        G, N, K = t.shape
        qT, eT = _mx_gpu("3d", t)
        h3 = host.reshape(G, N, K)
        spans = [(g, n0, n1) for g in range(G) for n0, n1 in _chunks(N, 2048)]
        results = oracle_map("mx_quant_1x32_col", [(np.ascontiguousarray(h3[g, n0:n1]),) for g, n0, n1 in spans])
        for (g, n0, n1), (qo, eo) in zip(spans, results):
            assert np.array_equal(qT[g][:, n0:n1], qo), ("w", "3d", g, n0)
            assert np.array_equal(eT[g][:, n0 // 32:n1 // 32], eo), ("w", "3d e8", g, n0)
            assert np.array_equal(fqT[g][:, n0:n1], qo), ("w", "fused 3d", g, n0)
            assert np.array_equal(feT[g][:, n0 // 32:n1 // 32], eo), ("w", "fused 3d e8", g, n0)


def test_selftest_bounded_wait_reports_timeout():
    B.fp8bw_selftest_bounded_wait(20000)          # 20 ms on a barrier nobody signals
    with pytest.raises(B.Fp8bwError) as e:
        B.fp8bw_sync_status()
    assert e.value.code == B.ERR_TIMEOUT
    B.fp8bw_sync_status()                          # the word was cleared; the context is usable
    x = adversarial_bf16(128, 128, 0)
    q, s = run_row(x)
    assert np.array_equal(q, oracle.quant_1x128_row(f32(x))[0])
