"""Pins of the oracle's blockwise quantizers and GEMMs.

Each check is fixed by the mathematics or by an independent computation, not
by re-running the oracle's own formula:
* hand blocks whose scale is an exact power of two, so ties stay exact ties;
* the invariant that every block's largest magnitude lands on +-448 exactly;
* the dequantization error bound of e4m3 round-to-nearest;
* all-zero and constant blocks;
* brute-force per-block loops on small inputs (indices and layouts);
* invariance under 128-aligned row/column sharding;
* GEMMs: an exact integer case with power-of-two scales computed blockwise in
  int64, an identity weight, and the SQNR level expected from e4m3 rounding.
"""
import numpy as np
import pytest

import oracle
from mxfp8_precision_gemms_fp8bw_gb300 import inputs


def _bf16(a) -> np.ndarray:
    """Round a float array to bf16 values (returned as float32) via torch."""
    import torch
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def test_eps_constant_and_scale_of_zero_block():
    assert oracle.EPS == np.float32(1e-12)
    x = np.zeros((128, 128), np.float32)
    q, s = oracle.quant_1x128_row(x)
    assert np.all(q == 0)
    assert s.dtype == np.float32
    # scale = fl32(1e-12) / 448 in float32
    assert np.all(s == np.float32(np.float32(1e-12) / np.float32(448.0)))


def test_hand_block_power_of_two_scale_exact_ties():
    # amax = 448 -> s = 1 exactly, so each value is rounded directly.
    row = np.zeros(128, np.float32)
    row[:7] = [448.0, 10.5, 11.5, 3 * 2.0 ** -10, 2.0 ** -10, -0.0, -248.0]
    x = np.tile(row, (128, 1))
    q, s = oracle.quant_1x128_row(x)
    assert np.all(s == 1.0)
    assert list(q[0, :7]) == [0x7E, 0x52, 0x54, 0x02, 0x00, 0x80, 0xF8]
    # amax = 448 * 2^-5 = 14 -> s = 2^-5; 14 * (10.5 / 448) = 0.328125 = 10.5 * 2^-5
    x2 = x * np.float32(2.0 ** -5)
    q2, s2 = oracle.quant_1x128_row(x2)
    assert np.all(s2 == np.float32(2.0 ** -5))
    assert np.array_equal(q2[:, :5], q[:, :5])


def test_quotient_is_a_division_not_a_reciprocal_multiply():
    # amax = 392 gives s = 392/448 = 0.875 exactly.  x = 1.3671875 (a bf16
    # value) gives x/s = 1.5625 exactly: the tie between 1.5 (0x3C, even
    # mantissa) and 1.625 (0x3D), so RNE picks 0x3C.  Multiplying by the
    # float32 reciprocal instead gives 1.5625001 and 0x3D.
    row = np.zeros(128, np.float32)
    row[0], row[1] = 392.0, 1.3671875
    q, s = oracle.quant_1x128_row(np.tile(row, (128, 1)))
    assert np.all(s == np.float32(0.875))
    assert np.all(q[:, 1] == 0x3C) and np.all(q[:, 0] == 0x7E)


def test_block_amax_maps_to_448_and_constant_block():
    rng = np.random.default_rng(0)
    x = _bf16(rng.standard_normal((256, 512)) * np.exp2(rng.integers(-20, 20, size=(256, 1))))
    q, s = oracle.quant_1x128_row(x)
    mags = np.abs(oracle.e4m3_decode(q)).reshape(256, 4, 128)
    assert np.all(mags.max(axis=2) == 448.0)
    # the element holding the amax is the one that encodes to +-448
    blocks = np.abs(x).reshape(256, 4, 128)
    arg = blocks.argmax(axis=2)
    assert np.all(np.take_along_axis(mags, arg[..., None], axis=2)[..., 0] == 448.0)
    c = np.full((128, 256), -3.25, np.float32)
    qc, sc = oracle.quant_1x128_row(c)
    assert np.all(qc == 0xFE)


def _dequant_bound_ok(x, deq, s_per_elem):
    x = x.astype(np.float64)
    bound = 2.0 ** -4 * np.abs(x) * (1 + 2.0 ** -18) + 2.0 ** -10 * s_per_elem
    return np.all(np.abs(deq - x) <= bound)


def test_dequant_error_bound_all_quantizers():
    rng = np.random.default_rng(1)
    x = _bf16(rng.standard_normal((384, 640)) * np.exp2(rng.uniform(-30, 30, size=(384, 1))))
    q, s = oracle.quant_1x128_row(x)
    deq = oracle.dequant_1x128_row(q, s)
    assert _dequant_bound_ok(x, deq, np.repeat(s.T.astype(np.float64), 128, axis=1))
    qT, sT = oracle.quant_1x128_col(x)
    degT = oracle.dequant_1x128_row(qT, sT)
    assert _dequant_bound_ok(x.T, degT, np.repeat(sT.T.astype(np.float64), 128, axis=1))
    qw, qwT, sw = oracle.quant_128x128(x)
    deqw = oracle.dequant_128x128(qw, sw)
    full = np.repeat(np.repeat(sw.astype(np.float64), 128, 0), 128, 1)
    assert _dequant_bound_ok(x, deqw, full)
    assert np.array_equal(qwT, qw.T)


def _brute_scale(block):
    amax = np.float32(0.0)
    for v in block.ravel():
        amax = max(amax, np.float32(abs(v)))
    return np.float32(max(amax, np.float32(1e-12)) / np.float32(448.0))


def test_brute_force_loops_layouts():
    rng = np.random.default_rng(2)
    x = _bf16(rng.standard_normal((256, 384)))
    R, C = x.shape
    q, s = oracle.quant_1x128_row(x)
    qT, sT = oracle.quant_1x128_col(x)
    qw, qwT, sw = oracle.quant_128x128(x)
    assert s.shape == (C // 128, R) and sT.shape == (R // 128, C) and sw.shape == (R // 128, C // 128)
    for r in (0, 77, 255):
        for kb in range(C // 128):
            blk = x[r, kb * 128:(kb + 1) * 128]
            sc = _brute_scale(blk)
            assert s[kb, r] == sc
            codes = oracle.e4m3_encode(np.array([np.float32(v / sc) for v in blk], np.float32))
            assert np.array_equal(q[r, kb * 128:(kb + 1) * 128], codes)
    for c in (0, 130, 383):
        for rb in range(R // 128):
            blk = x[rb * 128:(rb + 1) * 128, c]
            sc = _brute_scale(blk)
            assert sT[rb, c] == sc
            codes = oracle.e4m3_encode(np.array([np.float32(v / sc) for v in blk], np.float32))
            assert np.array_equal(qT[c, rb * 128:(rb + 1) * 128], codes)
    for rb in range(R // 128):
        for cb in range(C // 128):
            tile = x[rb * 128:(rb + 1) * 128, cb * 128:(cb + 1) * 128]
            assert sw[rb, cb] == _brute_scale(tile)


def test_sharding_invariance():
    rng = np.random.default_rng(3)
    x = _bf16(rng.standard_normal((512, 512)) * 3)
    q, s = oracle.quant_1x128_row(x)
    qa, sa = oracle.quant_1x128_row(np.ascontiguousarray(x[:256]))
    qb, sb = oracle.quant_1x128_row(np.ascontiguousarray(x[256:]))
    assert np.array_equal(q, np.concatenate([qa, qb], 0)) and np.array_equal(s, np.concatenate([sa, sb], 1))
    qc, sc = oracle.quant_1x128_row(np.ascontiguousarray(x[:, :128]))
    assert np.array_equal(q[:, :128], qc) and np.array_equal(s[:1], sc)
    qw, _, sw = oracle.quant_128x128(x)
    qw2, _, sw2 = oracle.quant_128x128(np.ascontiguousarray(x[128:384, 256:]))
    assert np.array_equal(qw[128:384, 256:], qw2) and np.array_equal(sw[1:3, 2:], sw2)


# ---------------------------------------------------------------- GEMMs

def _int_codes(rng, shape, lo=-8, hi=8):
    """e4m3 codes of small integers (all exactly representable) and their values."""
    vals = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return oracle.e4m3_encode(vals), vals.astype(np.int64)


def test_gemm_fwd_exact_integer_blockwise():
    # Codes hold small integers; scales are distinct powers of two per block,
    # so every partial sum is exact and the expected value can be formed
    # blockwise in int64 -- the per-128-K structure of the method, written
    # independently of the oracle's dequantize-then-matmul.
    rng = np.random.default_rng(4)
    M, N, K = 128, 256, 384
    xq, xi = _int_codes(rng, (M, K))
    wq, wi = _int_codes(rng, (N, K))
    xs = np.exp2(rng.integers(-6, 6, size=(K // 128, M))).astype(np.float32)
    ws = np.exp2(rng.integers(-6, 6, size=(N // 128, K // 128))).astype(np.float32)
    want = np.zeros((M, N), np.float64)
    for kb in range(K // 128):
        part = xi[:, kb * 128:(kb + 1) * 128] @ wi[:, kb * 128:(kb + 1) * 128].T   # int64 exact
        for nb in range(N // 128):
            want[:, nb * 128:(nb + 1) * 128] += (part[:, nb * 128:(nb + 1) * 128]
                                                 * xs[kb][:, None].astype(np.float64) * float(ws[nb, kb]))
    got = oracle.gemm_fwd(xq, xs, wq, ws)
    assert np.array_equal(got, want)


def test_gemm_dgrad_and_wgrad_exact_integer_blockwise():
    rng = np.random.default_rng(5)
    M, N, K = 256, 256, 384
    dyq, dyi = _int_codes(rng, (M, N))
    wq, wi = _int_codes(rng, (N, K))
    dys = np.exp2(rng.integers(-6, 6, size=(N // 128, M))).astype(np.float32)
    ws = np.exp2(rng.integers(-6, 6, size=(N // 128, K // 128))).astype(np.float32)
    want = np.zeros((M, K), np.float64)
    for nb in range(N // 128):
        part = dyi[:, nb * 128:(nb + 1) * 128] @ wi[nb * 128:(nb + 1) * 128, :]
        for kb in range(K // 128):
            want[:, kb * 128:(kb + 1) * 128] += (part[:, kb * 128:(kb + 1) * 128]
                                                 * dys[nb][:, None].astype(np.float64) * float(ws[nb, kb]))
    assert np.array_equal(oracle.gemm_dgrad(dyq, dys, wq, ws), want)

    # wgrad: both operands colwise along M (1x128 blocks along tokens).
    dyqT, dyTi = _int_codes(rng, (N, M))
    xqT, xTi = _int_codes(rng, (K, M))
    dysT = np.exp2(rng.integers(-6, 6, size=(M // 128, N))).astype(np.float32)
    xsT = np.exp2(rng.integers(-6, 6, size=(M // 128, K))).astype(np.float32)
    want = np.zeros((N, K), np.float64)
    for mb in range(M // 128):
        part = dyTi[:, mb * 128:(mb + 1) * 128] @ xTi[:, mb * 128:(mb + 1) * 128].T
        want += part * np.outer(dysT[mb].astype(np.float64), xsT[mb].astype(np.float64))
    assert np.array_equal(oracle.gemm_wgrad(dyqT, dysT, xqT, xsT), want)


def test_gemm_identity_weight():
    rng = np.random.default_rng(6)
    x = _bf16(rng.standard_normal((128, 256)))
    xq, xs = oracle.quant_1x128_row(x)
    wq = oracle.e4m3_encode(np.eye(256, dtype=np.float32) * 448.0)
    ws = np.ones((2, 2), np.float32)
    y = oracle.gemm_fwd(xq, xs, wq, ws)
    assert np.array_equal(y, oracle.dequant_1x128_row(xq, xs) * 448.0)


def test_linear_sqnr_matches_e4m3_rounding_level():
    # e4m3 RNE with 3 mantissa bits gives roughly 10 log10(12 * 2^8) ~ 35 dB per
    # operand for uniformly spread mantissas; a GEMM of two quantized operands
    # lands near 30 dB.  The bound the tests apply is 25 dB.
    t = inputs.tiny()
    x = inputs.bf16_to_f32_numpy(t.x)
    w = inputs.bf16_to_f32_numpy(t.w)
    dy = inputs.bf16_to_f32_numpy(t.dy)
    xq, xs = oracle.quant_1x128_row(x)
    wq, wqT, ws = oracle.quant_128x128(w)
    y = oracle.gemm_fwd(xq, xs, wq, ws)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    snr = oracle.sqnr_db(ref, y)
    assert 27.0 < snr < 40.0, snr
    dyq, dys = oracle.quant_1x128_row(dy)
    dx = oracle.gemm_dgrad(dyq, dys, wq, ws)
    assert 27.0 < oracle.sqnr_db(dy.astype(np.float64) @ w.astype(np.float64), dx) < 40.0
    dyqT, dysT = oracle.quant_1x128_col(dy)
    xqT, xsT = oracle.quant_1x128_col(x)
    dW = oracle.gemm_wgrad(dyqT, dysT, xqT, xsT)
    assert 27.0 < oracle.sqnr_db(dy.astype(np.float64).T @ x.astype(np.float64), dW) < 40.0


def test_metrics_closed_forms():
    ref = np.linspace(-3, 5, 1000)
    assert oracle.sqnr_db(ref, ref * (1 + 1e-2)) == pytest.approx(40.0, abs=1e-9)
    assert oracle.sqnr_db(ref, ref) == float("inf")
    a = np.array([[3.0, 4.0], [0.0, 0.0]])
    assert np.allclose(oracle.row_norms(a), [5.0, 0.0])
    err = oracle.normalized_gemm_error(np.array([[1.0, 0.0]]), np.array([[0.5, 0.0]]), [2.0], [0.5, 0.0], 0.0)
    assert err[0, 0] == 0.5 and err[0, 1] == 0.0
    # with the bf16 allowance the first 2^-8 * |ref| of the difference is free
    err = oracle.normalized_gemm_error(np.array([[1.0]]), np.array([[0.5]]), [2.0], [0.5])
    assert err[0, 0] == (0.5 - 0.5 / 256) / 1.0
    err2 = oracle.normalized_gemm_error(np.array([[0.0, 1e-9]]), np.zeros((1, 2)), [2.0], [0.5, 0.0])
    assert err2[0, 1] == np.inf


def test_bf16_allowance_is_the_format_unit_roundoff():
    # bf16 has 8 significant bits: next to 64 its spacing is 0.5, so the
    # correctly rounded bf16 of -67.7497 is -67.5, off by 0.2497 = 0.00369 |C|:
    # inside 2^-8 |C| (the allowance), beyond 2^-9 |C|.
    import torch
    c = -67.74966269465418
    r = float(torch.tensor(c, dtype=torch.float64).to(torch.bfloat16).to(torch.float64))
    assert r == -67.5
    assert 2.0 ** -9 * abs(c) < abs(r - c) <= oracle.BF16_ROUNDOFF * abs(c)
    # the rounding of every bf16-representable neighbourhood stays within the allowance
    xs = np.linspace(1.0, 2.0, 100001) * 2.0 ** 5
    rb = torch.from_numpy(xs).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.all(np.abs(rb - xs) <= oracle.BF16_ROUNDOFF * np.abs(xs))
    # one bf16 ulp beyond the correctly rounded value is not free: a 2^-7 |C| miss on
    # parallel operands (|C| = |a||b|) fails the 2e-3 bar
    assert oracle.normalized_gemm_error(np.array([[c * (1 + 2.0 ** -7)]]), np.array([[c]]), [abs(c)], [1.0])[0, 0] \
        > oracle.GEMM_TOL
