"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each.

Every mutation below is applied with monkeypatch for the duration of one
pin; the pin must then fail.  This shows the pins are sharp enough to catch a
dropped term, a wrong constant, a reciprocal multiply in place of the
division, a transposed scale index, or a wrong rounding rule.
"""
import numpy as np
import pytest

import oracle
import oracle.blockwise as ob
import oracle.e4m3 as oe
import oracle.mx as om

import test_oracle_blockwise as tb
import test_oracle_e4m3 as te
import test_oracle_mx as tm

FAIL = (AssertionError, ValueError, IndexError)


def _expect_fail(fn):
    with pytest.raises(FAIL):
        fn()


def test_wrong_max_constant_is_caught(monkeypatch):
    monkeypatch.setattr(ob, "block_scale",
                        lambda amax: (np.maximum(np.asarray(amax, np.float32), ob.EPS) / np.float32(447.0)).astype(np.float32))
    _expect_fail(tb.test_hand_block_power_of_two_scale_exact_ties)


def test_missing_eps_floor_is_caught(monkeypatch):
    monkeypatch.setattr(ob, "block_scale",
                        lambda amax: (np.asarray(amax, np.float32) / np.float32(448.0)).astype(np.float32))
    with np.errstate(divide="ignore", invalid="ignore"):
        _expect_fail(tb.test_eps_constant_and_scale_of_zero_block)


def test_reciprocal_multiply_is_caught(monkeypatch):
    def recip(x, s):
        r = (np.float32(1.0) / s).astype(np.float32)
        return oe.e4m3_encode((x * r).astype(np.float32))
    monkeypatch.setattr(ob, "quantize_with_scale", recip)
    _expect_fail(tb.test_quotient_is_a_division_not_a_reciprocal_multiply)


def test_transposed_weight_scale_is_caught(monkeypatch):
    orig = ob.dequant_128x128
    monkeypatch.setattr(ob, "dequant_128x128", lambda q, s: orig(q, np.ascontiguousarray(np.asarray(s)[::-1])))
    _expect_fail(tb.test_gemm_fwd_exact_integer_blockwise)


def test_wrong_activation_scale_index_is_caught(monkeypatch):
    orig = ob.dequant_1x128_row
    monkeypatch.setattr(ob, "dequant_1x128_row", lambda q, s: orig(q, np.roll(np.asarray(s), 1, axis=1)))
    _expect_fail(tb.test_gemm_dgrad_and_wgrad_exact_integer_blockwise)


def test_round_half_away_is_caught(monkeypatch):
    real_rint = np.rint

    class _NP:
        def __getattr__(self, name):
            if name == "rint":
                return lambda a: np.floor(np.asarray(a) + 0.5)
            return getattr(np, name)
    monkeypatch.setattr(oe, "np", _NP())
    try:
        _expect_fail(te.test_golden_rounding_cases)
    finally:
        assert real_rint is np.rint


def test_no_saturation_is_caught(monkeypatch):
    orig = oe.e4m3_encode

    def nosat(v):
        c = orig(v)
        a = np.abs(np.asarray(v, np.float64))
        return np.where(a >= 464.0, c | 0x7F, c).astype(np.uint8)
    monkeypatch.setattr(oracle, "e4m3_encode", nosat)
    _expect_fail(te.test_golden_rounding_cases)


def test_exponent_off_by_one_is_caught(monkeypatch):
    orig = om.e8m0_exponent
    monkeypatch.setattr(oracle, "e8m0_exponent", lambda a, mode: orig(a, mode) + (mode == om.RCEIL))
    _expect_fail(tm.test_golden_exponents)


def test_group_boundary_off_by_block_is_caught(monkeypatch):
    orig = om.group_starts
    monkeypatch.setattr(om, "group_starts", lambda ge: orig(ge) + 32 * (np.arange(len(ge)) > 0))
    _expect_fail(tm.test_grouped_wgrad_sums_to_full_contraction_and_empty_is_zero)
