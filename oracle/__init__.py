"""fp64 CPU oracle for the RMSNorm family (plain, fused with RoPE, AdaLN,
residual add), standalone RoPE from positions, and tanh GELU / GEGLU --
TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it, and this package imports nothing from
the product path: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, binary64, sequential sums); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
bfloat16 tensors travel as ``numpy.uint16`` arrays of bit patterns; every
operation also takes ``numpy.float16`` (IEEE binary16) and ``numpy.float32``
arrays, the pages' other two precision modes, and answers in the same type.

Definition followed (the pages print no formula; see ``oracle.c`` for the
page sections cited):
    n_j = x_j * w_j / sqrt(mean(x^2) + eps), then per-head RoPE
    a' = a c - b s, b' = a s + b c, rounded once to bfloat16 (RNE).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

INTERLEAVED = 0
SPLIT_HALF = 1

# element formats (the codes of oracle.c)
FMT_BF16, FMT_F16, FMT_F32 = 0, 1, 2
_FMT_OF_DTYPE = {np.dtype(np.uint16): FMT_BF16, np.dtype(np.float16): FMT_F16,
                 np.dtype(np.float32): FMT_F32}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, -O2).

    ``-ffp-contract=off`` keeps every multiply and add separately rounded on
    both x86-64 and AArch64 hosts.
    """
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            lib.oracle_widen_bf16.argtypes = [P, P, I64]
            lib.oracle_widen_bf16.restype = None
            lib.oracle_round_bf16.argtypes = [P, P, I64]
            lib.oracle_round_bf16.restype = None
            lib.oracle_rms_norm.argtypes = [P, P, P, I64, I64, ctypes.c_float, P]
            lib.oracle_rms_norm.restype = ctypes.c_int
            lib.oracle_rms_norm_rope.argtypes = [
                P, P, P, P, P, I64, I64, I64, ctypes.c_int, ctypes.c_float,
                I64, I64, P]
            lib.oracle_rms_norm_rope.restype = ctypes.c_int
            lib.oracle_rms_norm_adaln.argtypes = [P, P, P, P, P, I64, I64, I64, I64,
                                                  ctypes.c_float, P]
            lib.oracle_rms_norm_adaln.restype = ctypes.c_int
            lib.oracle_add_rms_norm.argtypes = [P, P, P, P, P, I64, I64, ctypes.c_float, P]
            lib.oracle_add_rms_norm.restype = ctypes.c_int
            I32, F32 = ctypes.c_int, ctypes.c_float
            lib.oracle_widen_fmt.argtypes = [I32, P, P, I64]
            lib.oracle_widen_fmt.restype = None
            lib.oracle_round_fmt.argtypes = [I32, P, P, I64]
            lib.oracle_round_fmt.restype = None
            lib.oracle_rms_norm_fmt.argtypes = [I32, P, P, P, I64, I64, F32, P]
            lib.oracle_rms_norm_fmt.restype = I32
            lib.oracle_rms_norm_rope_fmt.argtypes = [I32, P, P, P, P, P, I64, I64, I64, I32,
                                                     F32, I64, I64, P]
            lib.oracle_rms_norm_rope_fmt.restype = I32
            lib.oracle_rms_norm_adaln_fmt.argtypes = [I32, P, P, P, P, P, I64, I64, I64, I64,
                                                      F32, P]
            lib.oracle_rms_norm_adaln_fmt.restype = I32
            lib.oracle_add_rms_norm_fmt.argtypes = [I32, P, P, P, P, P, I64, I64, F32, P]
            lib.oracle_add_rms_norm_fmt.restype = I32
            lib.oracle_rope_positions.argtypes = [I32, P, P, I64, I64, I64, I32, I64, I64, I64,
                                                  I64, I64, I64, ctypes.c_double, I64, P]
            lib.oracle_rope_positions.restype = I32
            lib.oracle_rope_tables.argtypes = [P, P, I64, I64, I64, I64, I64, I64, I64, I64,
                                               ctypes.c_double]
            lib.oracle_rope_tables.restype = I32
            lib.oracle_gelu_tanh_fmt.argtypes = [I32, P, P, I64, P]
            lib.oracle_gelu_tanh_fmt.restype = None
            lib.oracle_geglu_fmt.argtypes = [I32, P, P, I64, I64, P]
            lib.oracle_geglu_fmt.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _u16(a, name):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"{name} must hold bfloat16 bit patterns as uint16")
    return a


def _elems(a, name, like=None):
    """(format code, contiguous array) of a bf16 (uint16 bits), float16 or
    float32 array; with ``like``, the array must have like's dtype."""
    a = np.ascontiguousarray(a)
    fmt = _FMT_OF_DTYPE.get(a.dtype)
    if fmt is None:
        raise TypeError(f"{name} must be uint16 (bfloat16 bits), float16 or float32")
    if like is not None and a.dtype != like.dtype:
        raise TypeError(f"{name} must have the dtype of x ({like.dtype})")
    return fmt, a


def widen(a: np.ndarray) -> np.ndarray:
    """Exact binary64 values of a bf16 (uint16 bits), float16 or float32 array."""
    fmt, a = _elems(a, "a")
    out = np.empty(a.shape, np.float64)
    _load().oracle_widen_fmt(fmt, _ptr(a), _ptr(out), a.size)
    return out


def round_to(values: np.ndarray, dtype) -> np.ndarray:
    """Round binary64 values once (RNE) to bf16 (``numpy.uint16`` bits),
    float16 or float32."""
    values = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(values.shape, dtype)
    fmt, out = _elems(out, "dtype")
    _load().oracle_round_fmt(fmt, _ptr(values), _ptr(out), values.size)
    return out


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """Exact binary64 values of bfloat16 bit patterns."""
    bits = _u16(bits, "bits")
    out = np.empty(bits.shape, np.float64)
    _load().oracle_widen_bf16(_ptr(bits), _ptr(out), bits.size)
    return out


def round_bf16(values: np.ndarray) -> np.ndarray:
    """Round binary64 values straight to bfloat16 (RNE); returns bit patterns."""
    values = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(values.shape, np.uint16)
    _load().oracle_round_bf16(_ptr(values), _ptr(out), values.size)
    return out


def _row_blocks(rows, threads):
    threads = max(1, min(threads, rows))
    step = -(-rows // threads)
    return [(r0, min(rows, r0 + step)) for r0 in range(0, rows, step)]


def rms_norm(x, w, eps, *, threads: int = 1, exact: bool = False):
    """Oracle RMSNorm over the last axis of ``x`` (uint16 bf16 bits, float16
    or float32; ``w`` of the same dtype).

    Returns the rounded values in x's dtype, or ``(values, exact_values)``
    when ``exact``.
    ``threads`` > 1 runs disjoint row ranges concurrently (ctypes releases the
    GIL during the call); the arithmetic per row is unchanged.
    """
    fmt, x = _elems(x, "x")
    H = x.shape[-1]
    rows = x.size // H if H else 0
    x2 = x.reshape(rows, H)
    w = None if w is None else _elems(w, "w", x)[1]
    if w is not None and w.size != H:
        raise ValueError("w must have hidden elements")
    y = np.empty_like(x2)
    ye = np.empty(x2.shape, np.float64) if exact else None
    lib = _load()

    def run(block):
        r0, r1 = block
        rc = lib.oracle_rms_norm_fmt(
            fmt, _ptr(y[r0:r1]), _ptr(x2[r0:r1]), _ptr(w), r1 - r0, H,
            ctypes.c_float(eps), None if ye is None else _ptr(ye[r0:r1]))
        if rc != 0:
            raise MemoryError("oracle_rms_norm failed")

    _run_blocks(run, rows, threads)
    y = y.reshape(x.shape)
    return (y, ye.reshape(x.shape)) if exact else y


def rms_norm_rope(x, w, cos, sin, heads, head_dim, mode, eps, *,
                  table_rows=None, threads: int = 1, exact: bool = False):
    """Oracle fused RMSNorm + RoPE.

    ``x``: [rows, heads*head_dim] (bf16 bits, float16 or float32);
    ``cos``/``sin``: float32
    [table_rows, head_dim/2]; row r uses table row ``r % table_rows``
    (``table_rows`` defaults to the tables' first dimension).
    """
    fmt, x = _elems(x, "x")
    H = heads * head_dim
    if x.shape[-1] != H:
        raise ValueError("last axis of x must be heads*head_dim")
    rows = x.size // H
    x2 = x.reshape(rows, H)
    w = None if w is None else _elems(w, "w", x)[1]
    cos = np.ascontiguousarray(cos, dtype=np.float32)
    sin = np.ascontiguousarray(sin, dtype=np.float32)
    P = head_dim // 2
    if table_rows is None:
        table_rows = cos.size // P
    if cos.size < table_rows * P or sin.size < table_rows * P:
        raise ValueError("tables too small")
    y = np.empty_like(x2)
    ye = np.empty(x2.shape, np.float64) if exact else None
    lib = _load()

    def run(block):
        r0, r1 = block
        rc = lib.oracle_rms_norm_rope_fmt(
            fmt, _ptr(y[r0:r1]), _ptr(x2[r0:r1]), _ptr(w), _ptr(cos), _ptr(sin),
            r1 - r0, heads, head_dim, mode, ctypes.c_float(eps), table_rows,
            r0, None if ye is None else _ptr(ye[r0:r1]))
        if rc != 0:
            raise RuntimeError(f"oracle_rms_norm_rope failed ({rc})")

    _run_blocks(run, rows, threads)
    y = y.reshape(x.shape)
    return (y, ye.reshape(x.shape)) if exact else y


def rms_norm_adaln(x, w, scale, shift, eps, *, rows_per_cond=None,
                   threads: int = 1, exact: bool = False):
    """Oracle AdaLN-modulated RMSNorm: norm(x) * w * (1 + scale) + shift.

    ``x``: [rows, H]; ``scale``/``shift``: [n_cond, H], all of one dtype
    (bf16 bits, float16 or float32); row r
    uses conditioning row ``r // rows_per_cond`` (default: rows / n_cond).
    """
    fmt, x = _elems(x, "x")
    H = x.shape[-1]
    rows = x.size // H
    x2 = x.reshape(rows, H)
    w = None if w is None else _elems(w, "w", x)[1]
    scale = _elems(scale, "scale", x)[1].reshape(-1, H)
    shift = _elems(shift, "shift", x)[1].reshape(-1, H)
    if scale.shape != shift.shape:
        raise ValueError("scale and shift must have the same shape")
    n_cond = scale.shape[0]
    if rows_per_cond is None:
        rows_per_cond = max(1, -(-rows // n_cond))
    if rows and (rows - 1) // rows_per_cond >= n_cond:
        raise ValueError("not enough conditioning rows")
    y = np.empty_like(x2)
    ye = np.empty(x2.shape, np.float64) if exact else None
    lib = _load()

    def run(block):
        r0, r1 = block
        rc = lib.oracle_rms_norm_adaln_fmt(
            fmt, _ptr(y[r0:r1]), _ptr(x2[r0:r1]), _ptr(w), _ptr(scale), _ptr(shift),
            r1 - r0, H, rows_per_cond, r0, ctypes.c_float(eps),
            None if ye is None else _ptr(ye[r0:r1]))
        if rc != 0:
            raise RuntimeError(f"oracle_rms_norm_adaln failed ({rc})")

    _run_blocks(run, rows, threads)
    y = y.reshape(x.shape)
    return (y, ye.reshape(x.shape)) if exact else y


def add_rms_norm(x, res, w, eps, *, threads: int = 1, exact: bool = False):
    """Oracle fused residual add + RMSNorm.

    Returns ``(y, h)`` in x's dtype (``h = round(x + res)``, ``y`` the
    RMSNorm of ``h``), or ``(y, h, y_exact)`` when ``exact``.
    """
    fmt, x = _elems(x, "x")
    res = _elems(res, "res", x)[1]
    if x.shape != res.shape:
        raise ValueError("x and res must have the same shape")
    H = x.shape[-1]
    rows = x.size // H if H else 0
    x2, r2 = x.reshape(rows, H), res.reshape(rows, H)
    w = None if w is None else _elems(w, "w", x)[1]
    y = np.empty_like(x2)
    h = np.empty_like(x2)
    ye = np.empty(x2.shape, np.float64) if exact else None
    lib = _load()

    def run(block):
        r0, r1 = block
        rc = lib.oracle_add_rms_norm_fmt(
            fmt, _ptr(y[r0:r1]), _ptr(h[r0:r1]), _ptr(x2[r0:r1]), _ptr(r2[r0:r1]), _ptr(w),
            r1 - r0, H, ctypes.c_float(eps), None if ye is None else _ptr(ye[r0:r1]))
        if rc != 0:
            raise MemoryError("oracle_add_rms_norm failed")

    _run_blocks(run, rows, threads)
    y, h = y.reshape(x.shape), h.reshape(x.shape)
    return (y, h, ye.reshape(x.shape)) if exact else (y, h)


def rope(x, heads, head_dim, mode, grid, pairs, theta=10000.0, *, threads: int = 1,
         exact: bool = False):
    """Oracle standalone RoPE with angles from token positions.

    ``x``: [rows, heads*head_dim] (bf16 bits, float16 or float32); row r is
    token ``r mod (T*H*W)`` of ``grid = (T, H, W)``; ``pairs = (nt, nh, nw)``
    split the head_dim/2 pairs over the axes (1D text: ``grid = (S, 1, 1)``,
    ``pairs = (head_dim/2, 0, 0)``).  Pair k of an axis with n pairs turns by
    ``coordinate * theta**(-k/n)``.
    """
    fmt, x = _elems(x, "x")
    HD = heads * head_dim
    if x.shape[-1] != HD:
        raise ValueError("last axis of x must be heads*head_dim")
    rows = x.size // HD
    x2 = x.reshape(rows, HD)
    y = np.empty_like(x2)
    ye = np.empty(x2.shape, np.float64) if exact else None
    T, H, W = grid
    nt, nh, nw = pairs
    lib = _load()

    def run(block):
        r0, r1 = block
        rc = lib.oracle_rope_positions(fmt, _ptr(y[r0:r1]), _ptr(x2[r0:r1]), r1 - r0, heads,
                                       head_dim, mode, T, H, W, nt, nh, nw, float(theta), r0,
                                       None if ye is None else _ptr(ye[r0:r1]))
        if rc != 0:
            raise RuntimeError(f"oracle_rope_positions failed ({rc})")

    _run_blocks(run, rows, threads)
    y = y.reshape(x.shape)
    return (y, ye.reshape(x.shape)) if exact else y


def rope_tables(tokens, head_dim, grid, pairs, theta=10000.0):
    """Oracle cos / sin tables ``[tokens, head_dim/2]`` (float64) of the
    angles of ``rope``: row s is token ``s mod (T*H*W)``."""
    P = head_dim // 2
    c = np.empty((tokens, P), np.float64)
    s = np.empty((tokens, P), np.float64)
    T, H, W = grid
    nt, nh, nw = pairs
    rc = _load().oracle_rope_tables(_ptr(c), _ptr(s), tokens, head_dim, T, H, W, nt, nh, nw,
                                    float(theta))
    if rc != 0:
        raise ValueError(f"oracle_rope_tables failed ({rc})")
    return c, s


def gelu_tanh(x, *, threads: int = 1, exact: bool = False):
    """Oracle tanh-approximated GELU, elementwise (uint16 bf16 bits, float16
    or float32; the result in the same dtype)."""
    fmt, x = _elems(x, "x")
    flat = x.reshape(-1)
    y = np.empty_like(flat)
    ye = np.empty(flat.shape, np.float64) if exact else None
    lib = _load()

    def run(block):
        r0, r1 = block
        lib.oracle_gelu_tanh_fmt(fmt, _ptr(y[r0:r1]), _ptr(flat[r0:r1]), r1 - r0,
                                 None if ye is None else _ptr(ye[r0:r1]))

    _run_blocks(run, flat.size, threads)
    y = y.reshape(x.shape)
    return (y, ye.reshape(x.shape)) if exact else y


def geglu(x, *, threads: int = 1, exact: bool = False):
    """Oracle GEGLU: x [..., 2h] -> [..., h], value * gelu(gate) with the
    value in the first half of the last axis and the gate in the second
    (uint16 bf16 bits, float16 or float32; the result in the same dtype)."""
    fmt, x = _elems(x, "x")
    h2 = x.shape[-1]
    if h2 % 2:
        raise ValueError("last axis must be even")
    h = h2 // 2
    rows = x.size // h2 if h2 else 0
    x2 = x.reshape(rows, h2)
    y = np.empty((rows, h), x.dtype)
    ye = np.empty((rows, h), np.float64) if exact else None
    lib = _load()

    def run(block):
        r0, r1 = block
        lib.oracle_geglu_fmt(fmt, _ptr(y[r0:r1]), _ptr(x2[r0:r1]), r1 - r0, h,
                             None if ye is None else _ptr(ye[r0:r1]))

    _run_blocks(run, rows, threads)
    shape = x.shape[:-1] + (h,)
    return (y.reshape(shape), ye.reshape(shape)) if exact else y.reshape(shape)


def _run_blocks(fn, rows, threads):
    if rows == 0:
        return
    blocks = _row_blocks(rows, threads)
    if len(blocks) == 1:
        fn(blocks[0])
        return
    with ThreadPoolExecutor(max_workers=len(blocks)) as ex:
        for f in [ex.submit(fn, b) for b in blocks]:
            f.result()
