"""Pins of the oracle's e4m3 codec against the format definition and independent codecs.

The codec is pinned (not merely re-run) by:
* hand-derived rounding cases (tests/golden/e4m3_rounding_cases.txt);
* torch's float8_e4m3fn type (and ml_dtypes', where installed): decode of all
  256 codes, and encode of every finite bf16 value and of crafted float32
  midpoints inside the range where neither library saturates differently;
* the round trip encode(decode(c)) == c over every non-NaN code.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn)
    return t.float().numpy().astype(np.float64)


def _torch_encode(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_golden_rounding_cases():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_rounding_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            val, code = line.split()[:2]
            rows.append((np.float32(float(val)), int(code, 16)))
    vals = np.array([r[0] for r in rows], dtype=np.float32)
    want = np.array([r[1] for r in rows], dtype=np.uint8)
    got = oracle.e4m3_encode(vals)
    assert np.array_equal(got, want), list(zip(vals, got, want))


def test_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = _torch_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert nan.sum() == 2                      # 0x7F and 0xFF only
    assert np.array_equal(mine[~nan], ref[~nan])
    # signed zero of 0x80
    assert np.signbit(mine[0x80]) and mine[0x80] == 0.0


def test_decode_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    codes = np.arange(256, dtype=np.uint8)
    ref = codes.view(ml.float8_e4m3fn).astype(np.float64)
    mine = oracle.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def test_format_landmarks():
    d = oracle.e4m3_decode(np.array([0x7E, 0x08, 0x07, 0x01, 0x38, 0x00], np.uint8))
    assert list(d) == [448.0, 2.0 ** -6, 7 * 2.0 ** -9, 2.0 ** -9, 1.0, 0.0]
    assert oracle.E4M3_MAX == 448.0


def test_roundtrip_every_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    back = oracle.e4m3_encode(oracle.e4m3_decode(codes).astype(np.float32))
    assert np.array_equal(back, codes)


def _all_finite_bf16_as_f32() -> np.ndarray:
    bits = np.arange(65536, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    return v[np.isfinite(v)]


def test_encode_every_bf16_matches_torch_in_range():
    v = _all_finite_bf16_as_f32()
    inside = np.abs(v) < 464.0             # torch turns values >= 464 into NaN (no saturation)
    mine = oracle.e4m3_encode(v[inside])
    ref = _torch_encode(v[inside])
    assert np.array_equal(mine, ref)
    # Outside, satfinite clamps every finite magnitude to 448 with its sign.
    out = v[~inside]
    got = oracle.e4m3_encode(out)
    want = np.where(np.signbit(out), 0xFE, 0x7E).astype(np.uint8)
    assert np.array_equal(got, want)


def test_encode_midpoints_and_neighbours_match_torch():
    # Every midpoint between adjacent e4m3 magnitudes (and the one between 0
    # and 2^-9), plus the float32 values one and two ulps either side.
    mags = np.unique(np.abs(oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))))
    mids = ((mags[:-1] + mags[1:]) / 2.0).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (mags[:-1] + mags[1:]) / 2.0)   # exact in fp32
    bits = mids.view(np.uint32).astype(np.int64)
    cand = np.concatenate([bits + d for d in (-2, -1, 0, 1, 2)]).astype(np.uint32).view(np.float32)
    cand = np.concatenate([cand, -cand])
    mine = oracle.e4m3_encode(cand)
    ref = _torch_encode(cand)
    assert np.array_equal(mine, ref)


def test_encode_random_float32_matches_torch():
    rng = np.random.default_rng(123)
    exps = rng.uniform(-14, 8.8, size=200000)
    v = (rng.choice([-1.0, 1.0], size=exps.size) * np.exp2(exps)).astype(np.float32)
    v = v[np.abs(v) < 464.0]
    assert np.array_equal(oracle.e4m3_encode(v), _torch_encode(v))


def test_encode_matches_ml_dtypes_saturating_cast():
    ml = pytest.importorskip("ml_dtypes")
    v = _all_finite_bf16_as_f32()
    v = v[np.abs(v) < 464.0]
    ref = v.astype(ml.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(oracle.e4m3_encode(v), ref)
