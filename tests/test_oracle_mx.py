"""Pins of the oracle's MXFP8 quantizers and grouped GEMMs.

* hand-derived E8M0 exponents (tests/golden/e8m0_exponent_cases.txt);
* exhaustive brute force of the exponent rule over every positive finite
  bf16 amax (search over E with exact float64 comparisons);
* ml_dtypes' float8_e8m0fnu decode of the biased byte, where installed;
* invariants: RCEIL puts each nonzero block's largest code in [224, 448],
  FLOOR puts the amax element in [256, 448]; dequantization is exact
  power-of-two scaling within e4m3's rounding bound;
* grouped GEMM: per-group brute force in int64 with power-of-two scales,
  empty groups give zeros, G = 1 equals the dense product, and the wgrad
  groups sum to the full-token contraction.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(a) -> np.ndarray:
    import torch
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def test_golden_exponents():
    with open(os.path.join(GOLDEN, "e8m0_exponent_cases.txt")) as f:
        rows = [l.split()[:3] for l in f if l.strip() and not l.startswith("#")]
    amax = np.array([float(r[0]) for r in rows], np.float32)
    assert list(oracle.e8m0_exponent(amax, oracle.RCEIL)) == [int(r[1]) for r in rows]
    assert list(oracle.e8m0_exponent(amax, oracle.FLOOR)) == [int(r[2]) for r in rows]


def _all_positive_finite_bf16() -> np.ndarray:
    bits = np.arange(1, 0x7F80, dtype=np.uint32) << 16
    return bits.view(np.float32)


def test_exponent_rule_exhaustive_over_bf16():
    a = _all_positive_finite_bf16().astype(np.float64)
    Es = np.arange(-200, 200)
    ok = np.ldexp(448.0, Es)[None, :] >= a[:, None]          # exact in float64
    brute_rceil = Es[np.argmax(ok, axis=1)]
    got = oracle.e8m0_exponent(a.astype(np.float32), oracle.RCEIL)
    assert np.array_equal(got, np.clip(brute_rceil, -127, 127))
    # FLOOR: 2^(E+8) <= amax < 2^(E+9) for every amax whose exponent is not clamped
    f = oracle.e8m0_exponent(a.astype(np.float32), oracle.FLOOR)
    inside = f > -127
    assert np.all(np.ldexp(1.0, f[inside] + 8) <= a[inside])
    assert np.all(a[inside] < np.ldexp(1.0, f[inside] + 9))
    assert np.all(a[~inside] < np.ldexp(1.0, -127 + 9))


def test_e8m0_byte_decodes_like_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    if not hasattr(ml, "float8_e8m0fnu"):
        pytest.skip("ml_dtypes without float8_e8m0fnu")
    rng = np.random.default_rng(0)
    x = _bf16(rng.standard_normal((64, 256)) * np.exp2(rng.integers(-60, 60, size=(64, 1))))
    q, e8 = oracle.mx_quant_1x32_row(x)
    scale = e8.view(ml.float8_e8m0fnu).astype(np.float64)
    assert np.array_equal(scale, np.ldexp(1.0, e8.astype(np.int64) - 127))


@pytest.mark.parametrize("mode", [oracle.RCEIL, oracle.FLOOR])
def test_mx_block_invariants(mode):
    rng = np.random.default_rng(1 + mode)
    x = _bf16(rng.standard_normal((96, 512)) * np.exp2(rng.integers(-40, 40, size=(96, 1))))
    x[5, :32] = 0.0
    q, e8 = oracle.mx_quant_1x32_row(x, mode)
    dec = oracle.e4m3_decode(q).reshape(96, 16, 32)
    blocks = np.abs(x).reshape(96, 16, 32)
    nz = blocks.max(axis=2) > 0
    top = np.abs(dec).max(axis=2)
    if mode == oracle.RCEIL:
        assert np.all((top[nz] >= 224) & (top[nz] <= 448))
    else:
        arg = blocks.argmax(axis=2)
        at = np.abs(np.take_along_axis(dec, arg[..., None], axis=2)[..., 0])
        assert np.all((at[nz] >= 256) & (at[nz] <= 448))
    assert e8[5, 0] == 0 and np.all(q[5, :32] & 0x7F == 0)
    # dequantization: dec(q) * 2^E within the e4m3 rounding bound of x
    deq = oracle.mx_dequant_row(q, e8)
    E = np.repeat(e8.astype(np.int64) - 127, 32, axis=1)
    bound = 2.0 ** -4 * np.abs(x) + np.ldexp(2.0 ** -10, E)
    sat = np.abs(x) * np.ldexp(1.0, -E) > 448.0        # FLOOR may saturate the top element
    assert np.all((np.abs(deq - x) <= bound) | sat)


def test_mx_col_and_3d_layouts():
    rng = np.random.default_rng(3)
    w = _bf16(rng.standard_normal((3, 64, 96)))
    qT, e8 = oracle.mx_quant_3d_col(w)
    assert qT.shape == (3, 96, 64) and e8.shape == (3, 96, 2)
    for g in range(3):
        for k in (0, 50, 95):
            for nb in range(2):
                col = w[g, nb * 32:(nb + 1) * 32, k]
                amax = np.abs(col).max()
                E = int(oracle.e8m0_exponent(np.array([amax], np.float32), oracle.RCEIL)[0])
                assert e8[g, k, nb] == E + 127
                codes = oracle.e4m3_encode((col * np.float32(2.0 ** -E)).astype(np.float32))
                assert np.array_equal(qT[g, k, nb * 32:(nb + 1) * 32], codes)


def _int_mx(rng, shape):
    vals = rng.integers(-8, 9, size=shape).astype(np.float32)
    e8 = (127 + rng.integers(-4, 5, size=shape[:-1] + (shape[-1] // 32,))).astype(np.uint8)
    return oracle.e4m3_encode(vals), e8, vals.astype(np.int64)


def _scaled_int(vals, e8):
    return vals.astype(np.float64) * np.ldexp(1.0, np.repeat(e8.astype(np.int64) - 127, 32, axis=-1))


def test_grouped_fwd_dgrad_brute_force_with_empty_group():
    rng = np.random.default_rng(4)
    M, N, K, G = 192, 64, 128, 4
    group_end = np.array([64, 64, 160, 192], np.int32)          # group 1 empty
    a, ae8, ai = _int_mx(rng, (M, K))
    b, be8, bi = _int_mx(rng, (G * N, K))
    got = oracle.mx_grouped_gemm(oracle.KIND_FWD, a, ae8, b, be8, group_end, G, M, N, K)
    starts = [0, 64, 64, 160]
    A = _scaled_int(ai, ae8)
    B = _scaled_int(bi, be8).reshape(G, N, K)
    for g in range(G):
        for m in range(starts[g], group_end[g]):
            for n in (0, 17, 63):
                want = sum(A[m, k] * B[g, n, k] for k in range(K))
                assert got[m, n] == want
    # DGRAD: b is [G, K_out, N_contract].  The whole output is pinned: every
    # row of every group against an int64 brute force of the group's own
    # expert (the values are integers times 2^E with E in [-4, 4], so each
    # operand times 2^4 is an exact integer and the product carries 2^8).
    a2, ae82, ai2 = _int_mx(rng, (M, N))
    b2, be82, bi2 = _int_mx(rng, (G * K, N))
    got2 = oracle.mx_grouped_gemm(oracle.KIND_DGRAD, a2, ae82, b2, be82, group_end, G, M, N, K)
    assert got2.shape == (M, K)
    A2 = ai2 << np.repeat(ae82.astype(np.int64) - 123, 32, axis=-1)
    B2 = (bi2 << np.repeat(be82.astype(np.int64) - 123, 32, axis=-1)).reshape(G, K, N)
    want = np.zeros((M, K), np.int64)
    for g in range(G):
        for m in range(starts[g], group_end[g]):
            for k in range(K):
                want[m, k] = int(np.sum(A2[m] * B2[g, k]))
    assert np.array_equal(got2 * 256.0, want.astype(np.float64))
    assert np.count_nonzero(want) > 0.9 * want.size           # the pin is not vacuous


def test_grouped_wgrad_sums_to_full_contraction_and_empty_is_zero():
    rng = np.random.default_rng(5)
    M, N, K, G = 256, 64, 96, 3
    group_end = np.array([96, 96, 256], np.int32)
    a, ae8, _ = _int_mx(rng, (N, M))
    b, be8, _ = _int_mx(rng, (K, M))
    dW = oracle.mx_grouped_gemm(oracle.KIND_WGRAD, a, ae8, b, be8, group_end, G, M, N, K)
    assert dW.shape == (G, N, K)
    assert np.all(dW[1] == 0.0)
    full = oracle.mx_dequant_row(a, ae8) @ oracle.mx_dequant_row(b, be8).T
    assert np.array_equal(dW.sum(axis=0), full)
    A = oracle.mx_dequant_row(a, ae8)
    B = oracle.mx_dequant_row(b, be8)
    assert dW[0, 7, 9] == sum(A[7, m] * B[9, m] for m in range(0, 96))


def test_grouped_single_group_is_dense():
    rng = np.random.default_rng(6)
    x = _bf16(rng.standard_normal((128, 256)))
    w = _bf16(rng.standard_normal((64, 256)) * 0.02)
    xq, xe = oracle.mx_quant_1x32_row(x)
    wq, we = oracle.mx_quant_1x32_row(w)
    y = oracle.mx_grouped_gemm(oracle.KIND_FWD, xq, xe, wq, we, np.array([128], np.int32), 1, 128, 64, 256)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    assert oracle.sqnr_db(ref, y) > 27.0
