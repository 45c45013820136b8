"""bf16 comparison for parity checks -- TEST INFRASTRUCTURE.

Tolerance: at most 1 bfloat16 ulp between the tested output and the
oracle's correctly rounded value, on every element.  It is measured as the
distance between the two bit patterns on the ordered integer line of
bfloat16 values (sign-magnitude mapped to a monotone integer, +0 and -0 both
at 0), which is well defined at binade edges and at zero.  A distance of 1
means the two values are neighbours; that happens when the exact value lies
within the test side's fp32 error of a rounding midpoint.
"""
from __future__ import annotations

import numpy as np


def ordinal(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def is_nan(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


def ulp_distance(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    return np.abs(ordinal(got) - ordinal(ref))


def compare_bf16(got: np.ndarray, ref: np.ndarray, max_ulps: int = 1) -> dict:
    """Element-by-element check; returns statistics and ``ok``."""
    got = np.asarray(got, dtype=np.uint16).reshape(-1)
    ref = np.asarray(ref, dtype=np.uint16).reshape(-1)
    if got.shape != ref.shape:
        raise ValueError(f"shape mismatch {got.shape} vs {ref.shape}")
    nan_mismatch = int(np.count_nonzero(is_nan(got) != is_nan(ref)))
    d = ulp_distance(got, ref)
    d = np.where(is_nan(got) & is_nan(ref), 0, d)
    worst = int(d.max()) if d.size else 0
    bad = np.flatnonzero(d > max_ulps)
    return {
        "elements": int(got.size),
        "exact": int(np.count_nonzero(d == 0)),
        "one_ulp": int(np.count_nonzero(d == 1)),
        "over_tolerance": int(bad.size),
        "max_ulps": worst,
        "nan_mismatch": nan_mismatch,
        "first_bad": [int(i) for i in bad[:8]],
        "ok": bad.size == 0 and nan_mismatch == 0,
    }


def widen(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def spacing_bf16(v: np.ndarray) -> np.ndarray:
    """Distance between adjacent bfloat16 values around |v| (8 significant
    bits; below 2^-126 the spacing stays 2^-133)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(a)
    e = np.maximum(e, -125)
    return np.ldexp(1.0, e - 8)


def compare_bf16_bounded(got: np.ndarray, exact: np.ndarray, bound: np.ndarray) -> dict:
    """Accept an element when it is within 1 ulp of the correctly rounded
    exact value, or when |got - exact| <= half a bf16 spacing (the test
    side's own final rounding) + ``bound`` (a bound on the test side's error
    before that rounding)."""
    got = np.asarray(got, dtype=np.uint16).reshape(-1)
    exact = np.asarray(exact, dtype=np.float64).reshape(-1)
    bound = np.asarray(bound, dtype=np.float64)
    bound = bound.reshape(-1) if bound.size == exact.size else np.broadcast_to(bound, exact.shape)
    g = widen(got)
    ref_bits = _round_bits(exact)
    d = ulp_distance(got, ref_bits)
    sp = np.maximum(spacing_bf16(g), spacing_bf16(exact))
    ok = (d <= 1) | (np.abs(g - exact) <= 0.5 * sp + bound)
    bad = np.flatnonzero(~ok)
    return {"elements": int(got.size), "exact": int(np.count_nonzero(d == 0)),
            "one_ulp": int(np.count_nonzero(d == 1)),
            "beyond_1ulp_within_bound": int(np.count_nonzero(ok & (d > 1))),
            "over_tolerance": int(bad.size), "first_bad": [int(i) for i in bad[:8]],
            "ok": bad.size == 0}


def _round_bits(v: np.ndarray) -> np.ndarray:
    # the oracle's own rounding (imported lazily: oracle builds a C library)
    import oracle
    return oracle.round_bf16(v)


# ---- float16 and float32 outputs (the pages' other precision modes) --------
#
# The same rule on the format's own bit patterns: ordinal distance (+0 and -0
# both at 0), NaN equal to NaN; spacing from the format's precision (binary16:
# 11 significant bits, fixed spacing 2^-24 below 2^-14; binary32: 24 bits,
# 2^-149 below 2^-126).

_FMT = {np.dtype(np.float16): (np.uint16, 11, -14), np.dtype(np.float32): (np.uint32, 24, -126)}


def _fmt_of(a):
    a = np.asarray(a)
    if a.dtype not in _FMT:
        raise TypeError("float16 or float32 expected")
    return a, _FMT[a.dtype]


def ordinal_fmt(a: np.ndarray) -> np.ndarray:
    a, (ut, prec, _) = _fmt_of(a)
    b = a.view(ut).astype(np.int64)
    top = 1 << (8 * np.dtype(ut).itemsize - 1)
    mag = b & (top - 1)
    return np.where(b & top, -mag, mag)


def spacing_fmt(v: np.ndarray, dtype) -> np.ndarray:
    _, prec, emin = _FMT[np.dtype(dtype)]
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(a)
    e = np.maximum(e, emin + 1)
    return np.ldexp(1.0, e - prec)


def compare_fmt(got: np.ndarray, ref: np.ndarray, max_ulps: int = 1) -> dict:
    """compare_bf16 for float16 / float32 arrays of the same dtype."""
    got, _ = _fmt_of(np.asarray(got).reshape(-1))
    ref, _ = _fmt_of(np.asarray(ref).reshape(-1))
    if got.dtype != ref.dtype or got.shape != ref.shape:
        raise ValueError("got and ref must have one dtype and shape")
    gn, rn = np.isnan(got), np.isnan(ref)
    d = np.abs(ordinal_fmt(got) - ordinal_fmt(ref))
    d = np.where(gn & rn, 0, d)
    bad = np.flatnonzero(d > max_ulps)
    return {"elements": int(got.size), "exact": int(np.count_nonzero(d == 0)),
            "one_ulp": int(np.count_nonzero(d == 1)), "over_tolerance": int(bad.size),
            "max_ulps": int(d.max()) if d.size else 0,
            "nan_mismatch": int(np.count_nonzero(gn != rn)),
            "first_bad": [int(i) for i in bad[:8]],
            "ok": bad.size == 0 and not np.any(gn != rn)}


def compare_fmt_bounded(got: np.ndarray, exact: np.ndarray, bound: np.ndarray) -> dict:
    """compare_bf16_bounded for float16 / float32 outputs: within 1 ulp of
    the correctly rounded exact value, or |got - exact| <= half a spacing +
    ``bound``."""
    import oracle
    got, _ = _fmt_of(np.asarray(got).reshape(-1))
    exact = np.asarray(exact, dtype=np.float64).reshape(-1)
    bound = np.asarray(bound, dtype=np.float64)
    bound = bound.reshape(-1) if bound.size == exact.size else np.broadcast_to(bound, exact.shape)
    ref = oracle.round_to(exact, got.dtype)
    d = np.abs(ordinal_fmt(got) - ordinal_fmt(ref))
    g = got.astype(np.float64)
    with np.errstate(invalid="ignore"):
        sp = np.maximum(spacing_fmt(g, got.dtype), spacing_fmt(exact, got.dtype))
        close = np.abs(g - exact) <= 0.5 * sp + bound
    ok = (d <= 1) | close | (np.isnan(g) & np.isnan(exact))
    bad = np.flatnonzero(~ok)
    return {"elements": int(got.size), "exact": int(np.count_nonzero(d == 0)),
            "one_ulp": int(np.count_nonzero(d == 1)),
            "beyond_1ulp_within_bound": int(np.count_nonzero(ok & (d > 1))),
            "over_tolerance": int(bad.size), "first_bad": [int(i) for i in bad[:8]],
            "ok": bad.size == 0}


def gelu_f32_bound(gate: np.ndarray, exact: np.ndarray, k0: float = 32.0) -> np.ndarray:
    """Error bound of an fp32 evaluation of value * gelu(gate) (value = 1
    for GELU), from the exact gate and the exact result:

        2^-24 (k0 + 5 |q| / (1 + 2^q)) |exact| + 2^-148,   k0 = 32,
        q = (2 / ln 2) sqrt(2 / pi) (gate + 0.044715 gate^3).

    Terms: q in fp32 carries a relative error of at most 6 * 2^-24 (the two
    constants' roundings, x^2, the fused multiply-add and the product), which
    moves s / (1 + s), s = 2^q, by the relative amount
    ln 2 * (1 - sigma) |dq| <= 4.2 * 2^-24 |q| / (1 + 2^q); the ex2 and rcp
    approximations and the remaining roundings are about 8 units of 2^-24,
    taken as k0 = 32 with margin; 2^-148 covers the rounding into the
    subnormal range (of gelu and then of the product)."""
    g = np.asarray(gate, dtype=np.float64)
    e = np.asarray(exact, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        q = (2.0 / np.log(2.0)) * np.sqrt(2.0 / np.pi) * (g + 0.044715 * g ** 3)
        left = np.exp(-np.logaddexp(0.0, q * np.log(2.0)))    # 1 / (1 + 2^q)
        rel = np.where(np.isfinite(q), k0 + 5.0 * np.abs(q) * left, np.inf)
        return np.ldexp(rel, -24) * np.abs(e) + 2.0 ** -148
