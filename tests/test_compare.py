"""The comparison rules the parity tests use (oracle/compare.py)."""
import numpy as np

import oracle
import synth
from oracle.compare import (compare_bf16, compare_bf16_bounded, ordinal, spacing_bf16,
                            ulp_distance)


def test_ordinal_is_monotone_over_all_finite_patterns():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = oracle.widen_bf16(b)
    fin = np.isfinite(v)
    order = np.argsort(v[fin], kind="stable")
    o = ordinal(b[fin])[order]
    assert np.all(np.diff(o) >= 0)
    assert ordinal(np.array([0x0000, 0x8000], np.uint16)).tolist() == [0, 0]


def test_one_ulp_rule():
    b = np.array([0x3F80, 0x3F80, 0x3F80, 0x0001], np.uint16)
    c = np.array([0x3F80, 0x3F81, 0x3F82, 0x8001], np.uint16)
    assert ulp_distance(b, c).tolist() == [0, 1, 2, 2]
    assert not compare_bf16(b, c)["ok"]
    assert compare_bf16(b[:2], c[:2])["ok"]


def test_spacing_matches_neighbours():
    b = np.arange(1, 0x7F7F, 997, dtype=np.uint32).astype(np.uint16)
    lo, hi = oracle.widen_bf16(b), oracle.widen_bf16((b + 1).astype(np.uint16))
    np.testing.assert_array_equal(spacing_bf16(lo), hi - lo)


def test_bounded_rule_accepts_rounding_and_rejects_errors():
    x = synth.normal_bf16(1, 0, 64 * 256).reshape(64, 256)
    sc = synth.normal_bf16(1, 3, 2 * 256, 0, 0.5).reshape(2, 256)
    sh = synth.normal_bf16(1, 4, 2 * 256, 0, 0.5).reshape(2, 256)
    y, ye = oracle.rms_norm_adaln(x, None, sc, sh, 1e-6, rows_per_cond=32, exact=True)
    bound = 1e-6 * np.abs(ye)
    assert compare_bf16_bounded(y, ye, bound)["ok"]
    # neighbours of the correctly rounded value are within 1 ulp
    assert compare_bf16_bounded((y.astype(np.int32) ^ 1).astype(np.uint16), ye, 0.0)["ok"]
    # three steps off is rejected unless the bound covers it
    off = (y.astype(np.int32) + 3).astype(np.uint16)
    assert compare_bf16_bounded(off, ye, bound)["over_tolerance"] > 0.99 * y.size
    # (three steps can cross a binade edge, where the spacing doubles)
    assert compare_bf16_bounded(off, ye, 8 * spacing_bf16(ye))["ok"]


def test_compare_fmt_neighbours_and_nan():
    from oracle.compare import compare_fmt
    for dt in (np.float16, np.float32):
        a = np.array([1.0, -2.0, 0.0, np.nan, 65000.0 if dt == np.float16 else 3e38], dt)
        b = np.nextafter(a, dt(np.inf)).astype(dt)
        b[3] = np.nan
        r = compare_fmt(b, a)
        assert r["ok"] and r["one_ulp"] == 4, r
        c = np.nextafter(b, dt(np.inf)).astype(dt)
        assert not compare_fmt(c, a)["ok"]
        assert compare_fmt(np.array([-0.0], dt), np.array([0.0], dt))["exact"] == 1
        assert not compare_fmt(np.array([np.nan], dt), np.array([1.0], dt))["ok"]


def test_compare_fmt_bounded_rejects_a_few_ulp_off():
    from oracle.compare import compare_fmt_bounded
    for dt in (np.float16, np.float32):
        exact = np.linspace(0.5, 3.0, 101)
        got = exact.astype(dt)
        assert compare_fmt_bounded(got, exact, 0.0)["ok"]
        off = got.copy()
        for _ in range(3):
            off = np.nextafter(off, dt(np.inf)).astype(dt)
        assert not compare_fmt_bounded(off, exact, 0.0)["ok"]
        # a bound of 4 spacings accepts them again
        sp = np.abs(np.nextafter(got, dt(np.inf)).astype(np.float64) - got)
        assert compare_fmt_bounded(off, exact, 4 * sp)["ok"]
