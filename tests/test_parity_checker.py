"""The comparison logic of ``parity`` on hand-made cases (CPU only).

The GPU tests trust these reports, so each rule is checked here: what counts
as within one bf16 ulp, when the cancellation allowance applies and is
counted, and how exponent bytes and e4m3 codes are compared.
"""
import math

import numpy as np
import pytest

import parity
from parity import Bf16Report, CacheReport, compare_cache


def _bits(values):
    v = np.asarray(values, np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)  # exact for bf16-representable values


def _report(gpu_values, exact, mag, oracle_values=None):
    rep = Bf16Report()
    oracle_values = exact if oracle_values is None else oracle_values
    rep.add(_bits(gpu_values), _bits(oracle_values), np.asarray(exact, np.float64),
            np.asarray(mag, np.float64))
    return rep


def test_ulp_of_bf16():
    assert parity.ulp_bf16(np.array([1.0]))[0] == 2.0 ** -7
    assert parity.ulp_bf16(np.array([1.5]))[0] == 2.0 ** -7
    assert parity.ulp_bf16(np.array([0.75]))[0] == 2.0 ** -8
    assert parity.ulp_bf16(np.array([0.0]))[0] == 2.0 ** -133
    assert parity.ulp_bf16(np.array([2.0 ** -130]))[0] == 2.0 ** -133


def test_one_ulp_passes_two_ulps_fail_without_cancellation():
    exact = 1.0 + 2.0 ** -9
    ok = _report([1.0 + 2.0 ** -7], [exact], [1.0], oracle_values=[1.0])
    ok.check()
    assert ok.beyond_ulp == 0 and ok.exact == 0
    bad = _report([1.0 + 2.0 ** -6], [exact], [1.0], oracle_values=[1.0])
    assert bad.bad == 1
    with pytest.raises(AssertionError):
        bad.check()


def test_cancellation_allowance_is_counted():
    # exact = 2^-10 formed from terms of magnitude 4: it cancels by 12 bits;
    # 3 ulps off (ulp = 2^-17) is 3 * 2^-17 < 2^-17 + 2^-15 * 4
    exact = 2.0 ** -10
    gpu = exact + 3 * 2.0 ** -17
    rep = _report([gpu], [exact], [4.0], oracle_values=[exact])
    rep.check()
    assert rep.beyond_ulp == 1
    assert rep.min_cancel_bits == pytest.approx(12.0)
    assert rep.max_ulps == pytest.approx(3.0)
    assert "1 beyond 1 ulp" in rep.summary()


def test_allowance_needs_a_cancellation():
    # the same absolute error with mag only 32x the result (5 bits) is refused
    exact = 2.0 ** -10
    gpu = exact + 3 * 2.0 ** -17
    rep = _report([gpu], [exact], [32 * exact], oracle_values=[exact])
    assert rep.bad == 1


def test_allowance_is_bounded():
    exact = 2.0 ** -10
    gpu = exact + 2.0 ** -12          # 32 ulps: beyond ulp + 2^-15 * 4
    rep = _report([gpu], [exact], [4.0], oracle_values=[exact])
    assert rep.bad == 1


def _cache_case(gpu_exp, ora_exp, margin, gpu_code=0x38, ora_code=0x38):
    g = np.zeros((2, 584), np.uint8)
    o = np.zeros((2, 584), np.uint8)
    g[1, 576] = gpu_exp
    o[1, 576] = ora_exp
    g[1, 5] = gpu_code
    o[1, 5] = ora_code
    slots = np.array([1], np.int64)
    ref = np.zeros((1, 512))
    mag = np.ones((1, 512))
    m = np.full((1, 7), math.inf)
    m[0, 0] = margin
    return compare_cache(g, o, slots, ref, mag, m)


def test_exponent_mismatch_only_at_a_near_tie():
    rep = _cache_case(120, 121, 2.0 ** -22)
    assert rep.exp_mismatch_ties == 1 and rep.exp_mismatch_bad == 0
    rep = _cache_case(120, 121, 2.0 ** -19)
    assert rep.exp_mismatch_bad == 1
    with pytest.raises(AssertionError):
        rep.check()


def test_codes_one_apart_allowed_two_apart_not():
    rep = _cache_case(120, 120, math.inf, gpu_code=0x39, ora_code=0x38)
    assert rep.codes_far == 0 and rep.codes_exact == rep.codes - 1
    rep = _cache_case(120, 120, math.inf, gpu_code=0x3A, ora_code=0x38)
    assert rep.codes_far == 1
    # +0 and -0 are the same code position; -0 and the smallest negative are one apart
    rep = _cache_case(120, 120, math.inf, gpu_code=0x80, ora_code=0x00)
    assert rep.codes_far == 0
    rep = _cache_case(120, 120, math.inf, gpu_code=0x81, ora_code=0x01)
    assert rep.codes_far == 1


def test_untouched_bytes_must_be_identical():
    g = np.zeros((3, 584), np.uint8)
    o = np.zeros((3, 584), np.uint8)
    g[2, 0] = 1                        # slot 2 is not mapped by any token
    with pytest.raises(AssertionError):
        compare_cache(g, o, np.array([1], np.int64), np.zeros((1, 512)), np.ones((1, 512)),
                      np.full((1, 7), math.inf))
