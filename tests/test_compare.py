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
