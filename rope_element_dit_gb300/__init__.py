"""Python binding of libltxk.so: RMSNorm and its fused forms (RoPE, AdaLN,
residual add) for bf16, fp16 and fp32 rows, and tanh GELU / GEGLU, on one
GB300 GPU.

The functions named ``ltxk_*`` mirror the C ABI in ``include/ltxk.h`` one to
one (integer device pointers in, an ``ltxk_status`` integer out).  The
``rms_norm`` / ``rms_norm_rope`` helpers marshal torch CUDA tensors into
those calls and raise :class:`LtxkError` on a non-zero status.  All
arithmetic runs in the library's CUDA kernels; there is no CPU path, and
importing this package fails if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libltxk.so")

OK = 0
ERR_NULL = 1
ERR_SHAPE = 2
ERR_ALIGN = 3
ERR_MODE = 4
ERR_OVERLAP = 5
ERR_CUDA = 6
ERR_TIMEOUT = 7
ERR_DTYPE = 8

DTYPE_BF16 = 0
DTYPE_F16 = 1
DTYPE_F32 = 2

PATH_AUTO = 0
PATH_REGISTERS = 1
PATH_TMA = 2

ROPE_INTERLEAVED = 0
ROPE_SPLIT_HALF = 1

OP_RMS_NORM = 0
OP_RMS_NORM_ROPE = 1
OP_RMS_NORM_ADALN = 2
OP_ADD_RMS_NORM = 3

KERNEL_NONE = 0
KERNEL_ROWS_VEC = 1
KERNEL_ROWS_ELEM = 2
KERNEL_ROWS_TMA = 3

__all__ = [
    # torch helpers (device tensors in, device tensors out)
    "rms_norm", "rms_norm_rope", "rms_norm_adaln", "add_rms_norm", "rope", "rope_tables",
    "gelu_tanh", "geglu", "rms_norm_host",
    # errors and constants
    "LtxkError", "Plan", "LIB_PATH", "EXPORTS",
    "OK", "ERR_NULL", "ERR_SHAPE", "ERR_ALIGN", "ERR_MODE", "ERR_OVERLAP", "ERR_CUDA",
    "ERR_TIMEOUT", "ERR_DTYPE", "ROPE_INTERLEAVED", "ROPE_SPLIT_HALF",
    "DTYPE_BF16", "DTYPE_F16", "DTYPE_F32", "PATH_AUTO", "PATH_REGISTERS", "PATH_TMA",
    "OP_RMS_NORM", "OP_RMS_NORM_ROPE", "OP_RMS_NORM_ADALN", "OP_ADD_RMS_NORM",
    "KERNEL_NONE", "KERNEL_ROWS_VEC", "KERNEL_ROWS_TMA", "KERNEL_ROWS_ELEM",
]

# Every entry point include/ltxk.h declares.
EXPORTS = ("ltxk_rms_norm", "ltxk_rms_norm_rope", "ltxk_rms_norm_rope_seq",
           "ltxk_rms_norm_adaln", "ltxk_rms_norm_host", "ltxk_add_rms_norm",
           "ltxk_fault_status", "ltxk_set_path", "ltxk_diag_missing_copy",
           "ltxk_rms_norm_noalloc", "ltxk_noalloc_fault_status",
           "ltxk_diag_noalloc_missing_copy", "ltxk_gelu_tanh", "ltxk_geglu",
           "ltxk_rms_norm_dt", "ltxk_rms_norm_rope_dt", "ltxk_rms_norm_adaln_dt",
           "ltxk_add_rms_norm_dt", "ltxk_plan_launch_dt", "ltxk_rope",
           "ltxk_gelu_tanh_dt", "ltxk_geglu_dt", "ltxk_rope_tables",
           "ltxk_status_string", "ltxk_last_cuda_error", "ltxk_plan_launch")
__all__ += list(EXPORTS)


class LtxkError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = f"{where}: {ltxk_status_string(status)} (status {status})"
        if status == ERR_CUDA:
            msg += f", cudaError {ltxk_last_cuda_error()}"
        super().__init__(msg)
        self.status = status


class Plan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("group_warps", ctypes.c_int),
                ("vec_per_lane", ctypes.c_int), ("block_threads", ctypes.c_int),
                ("rows_per_cta", ctypes.c_int), ("stages", ctypes.c_int),
                ("smem_bytes", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first with "
            "`python rope_element_dit_gb300/build.py` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I32, F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.ltxk_rms_norm.argtypes = [P, P, P, I64, I64, F32, P]
    lib.ltxk_rms_norm_rope.argtypes = [P, P, P, P, P, I64, I32, I32, I32, F32, P]
    lib.ltxk_rms_norm_rope_seq.argtypes = [P, P, P, P, P, I64, I32, I32, I32, F32, I64, P]
    for f in ("ltxk_rms_norm", "ltxk_rms_norm_rope", "ltxk_rms_norm_rope_seq"):
        getattr(lib, f).restype = I32
    lib.ltxk_rms_norm_adaln.argtypes = [P, P, P, P, P, I64, I64, I64, F32, P]
    lib.ltxk_rms_norm_adaln.restype = I32
    lib.ltxk_add_rms_norm.argtypes = [P, P, P, P, P, I64, I64, F32, P]
    lib.ltxk_add_rms_norm.restype = I32
    lib.ltxk_rms_norm_host.argtypes = [P, P, P, I64, I64, F32, P, I64,
                                       ctypes.POINTER(ctypes.c_void_p), I32]
    lib.ltxk_rms_norm_host.restype = I32
    lib.ltxk_rms_norm_noalloc.argtypes = [P, P, P, I64, I64, F32, P]
    lib.ltxk_rms_norm_noalloc.restype = I32
    lib.ltxk_noalloc_fault_status.argtypes = []
    lib.ltxk_noalloc_fault_status.restype = I32
    lib.ltxk_diag_noalloc_missing_copy.argtypes = [P, P, I64, I64, ctypes.c_uint64, P]
    lib.ltxk_diag_noalloc_missing_copy.restype = I32
    lib.ltxk_rms_norm_dt.argtypes = [P, P, P, I64, I64, F32, I32, P]
    lib.ltxk_rms_norm_rope_dt.argtypes = [P, P, P, P, P, I64, I32, I32, I32, F32, I64, I32, P]
    lib.ltxk_rms_norm_adaln_dt.argtypes = [P, P, P, P, P, I64, I64, I64, F32, I32, P]
    lib.ltxk_add_rms_norm_dt.argtypes = [P, P, P, P, P, I64, I64, F32, I32, P]
    for f in ("ltxk_rms_norm_dt", "ltxk_rms_norm_rope_dt", "ltxk_rms_norm_adaln_dt",
              "ltxk_add_rms_norm_dt"):
        getattr(lib, f).restype = I32
    lib.ltxk_plan_launch_dt.argtypes = [I32, I32, I64, I64, I32, I32, I32, ctypes.POINTER(Plan)]
    lib.ltxk_plan_launch_dt.restype = I32
    lib.ltxk_rope.argtypes = [P, P, I64, I32, I32, I32, I64, I64, I64, I32, I32, I32,
                              ctypes.c_double, I32, P]
    lib.ltxk_rope.restype = I32
    lib.ltxk_gelu_tanh.argtypes = [P, P, I64, P]
    lib.ltxk_gelu_tanh.restype = I32
    lib.ltxk_geglu.argtypes = [P, P, I64, I64, P]
    lib.ltxk_geglu.restype = I32
    lib.ltxk_rope_tables.argtypes = [P, P, I64, I32, I64, I64, I64, I32, I32, I32,
                                     ctypes.c_double, P]
    lib.ltxk_rope_tables.restype = I32
    lib.ltxk_gelu_tanh_dt.argtypes = [P, P, I64, I32, P]
    lib.ltxk_gelu_tanh_dt.restype = I32
    lib.ltxk_geglu_dt.argtypes = [P, P, I64, I64, I32, P]
    lib.ltxk_geglu_dt.restype = I32
    lib.ltxk_fault_status.argtypes = []
    lib.ltxk_fault_status.restype = I32
    lib.ltxk_set_path.argtypes = [I32]
    lib.ltxk_set_path.restype = I32
    lib.ltxk_diag_missing_copy.argtypes = [P, P, I64, I64, ctypes.c_uint64, P]
    lib.ltxk_diag_missing_copy.restype = I32
    lib.ltxk_status_string.argtypes = [I32]
    lib.ltxk_status_string.restype = ctypes.c_char_p
    lib.ltxk_last_cuda_error.argtypes = []
    lib.ltxk_last_cuda_error.restype = I32
    lib.ltxk_plan_launch.argtypes = [I32, I64, I64, I32, I32, I32, ctypes.POINTER(Plan)]
    lib.ltxk_plan_launch.restype = I32
    return lib


_lib = _load()


# ---- the C ABI, same names -------------------------------------------------

def ltxk_rms_norm(out, x, w, rows, hidden, eps, stream) -> int:
    return _lib.ltxk_rms_norm(out, x, w, rows, hidden, eps, stream)


def ltxk_rms_norm_rope(out, x, w, cos, sin, rows, heads, head_dim, mode, eps,
                       stream) -> int:
    return _lib.ltxk_rms_norm_rope(out, x, w, cos, sin, rows, heads, head_dim,
                                   mode, eps, stream)


def ltxk_rms_norm_rope_seq(out, x, w, cos, sin, rows, heads, head_dim, mode,
                           eps, seq_len, stream) -> int:
    return _lib.ltxk_rms_norm_rope_seq(out, x, w, cos, sin, rows, heads,
                                       head_dim, mode, eps, seq_len, stream)


def ltxk_rms_norm_adaln(out, x, w, scale, shift, rows, hidden, rows_per_cond, eps,
                        stream) -> int:
    return _lib.ltxk_rms_norm_adaln(out, x, w, scale, shift, rows, hidden, rows_per_cond,
                                    eps, stream)


def ltxk_add_rms_norm(out, residual_out, x, residual, w, rows, hidden, eps, stream) -> int:
    return _lib.ltxk_add_rms_norm(out, residual_out, x, residual, w, rows, hidden, eps, stream)


def ltxk_rms_norm_host(out_host, x_host, w, rows, hidden, eps, staging, staging_bytes,
                       streams, n_streams) -> int:
    """``streams``: a sequence of stream handles (ints), marshalled to an array."""
    arr = (ctypes.c_void_p * max(1, len(streams)))(*streams)
    return _lib.ltxk_rms_norm_host(out_host, x_host, w, rows, hidden, eps, staging,
                                   staging_bytes, arr, n_streams)


def ltxk_rms_norm_noalloc(out, x, w, rows, hidden, eps, stream) -> int:
    return _lib.ltxk_rms_norm_noalloc(out, x, w, rows, hidden, eps, stream)


def ltxk_rms_norm_dt(out, x, w, rows, hidden, eps, dtype, stream) -> int:
    return _lib.ltxk_rms_norm_dt(out, x, w, rows, hidden, eps, dtype, stream)


def ltxk_rms_norm_rope_dt(out, x, w, cos, sin, rows, heads, head_dim, mode, eps, seq_len,
                          dtype, stream) -> int:
    return _lib.ltxk_rms_norm_rope_dt(out, x, w, cos, sin, rows, heads, head_dim, mode, eps,
                                      seq_len, dtype, stream)


def ltxk_rms_norm_adaln_dt(out, x, w, scale, shift, rows, hidden, rows_per_cond, eps, dtype,
                           stream) -> int:
    return _lib.ltxk_rms_norm_adaln_dt(out, x, w, scale, shift, rows, hidden, rows_per_cond,
                                       eps, dtype, stream)


def ltxk_add_rms_norm_dt(out, residual_out, x, residual, w, rows, hidden, eps, dtype,
                         stream) -> int:
    return _lib.ltxk_add_rms_norm_dt(out, residual_out, x, residual, w, rows, hidden, eps, dtype,
                                     stream)


def ltxk_plan_launch_dt(op, dtype, rows, hidden, head_dim, mode, vector_ok):
    """Returns (status, Plan)."""
    p = Plan()
    st = _lib.ltxk_plan_launch_dt(op, dtype, rows, hidden, head_dim, mode,
                                  1 if vector_ok else 0, ctypes.byref(p))
    return st, p


def ltxk_rope(out, x, rows, heads, head_dim, mode, grid_t, grid_h, grid_w, pairs_t, pairs_h,
              pairs_w, theta, dtype, stream) -> int:
    return _lib.ltxk_rope(out, x, rows, heads, head_dim, mode, grid_t, grid_h, grid_w, pairs_t,
                          pairs_h, pairs_w, theta, dtype, stream)


def ltxk_gelu_tanh(out, x, n, stream) -> int:
    return _lib.ltxk_gelu_tanh(out, x, n, stream)


def ltxk_geglu(out, x, rows, hidden, stream) -> int:
    return _lib.ltxk_geglu(out, x, rows, hidden, stream)


def ltxk_rope_tables(cos_out, sin_out, tokens, head_dim, grid_t, grid_h, grid_w, pairs_t,
                     pairs_h, pairs_w, theta, stream) -> int:
    return _lib.ltxk_rope_tables(cos_out, sin_out, tokens, head_dim, grid_t, grid_h, grid_w,
                                 pairs_t, pairs_h, pairs_w, theta, stream)


def ltxk_gelu_tanh_dt(out, x, n, dtype, stream) -> int:
    return _lib.ltxk_gelu_tanh_dt(out, x, n, dtype, stream)


def ltxk_geglu_dt(out, x, rows, hidden, dtype, stream) -> int:
    return _lib.ltxk_geglu_dt(out, x, rows, hidden, dtype, stream)


def ltxk_fault_status() -> int:
    return _lib.ltxk_fault_status()


def ltxk_noalloc_fault_status() -> int:
    return _lib.ltxk_noalloc_fault_status()


def ltxk_diag_noalloc_missing_copy(out, x, rows, hidden, wait_limit_ns, stream) -> int:
    return _lib.ltxk_diag_noalloc_missing_copy(out, x, rows, hidden, wait_limit_ns, stream)


def ltxk_set_path(path: int) -> int:
    return _lib.ltxk_set_path(path)


def ltxk_diag_missing_copy(out, x, rows, hidden, wait_limit_ns, stream) -> int:
    return _lib.ltxk_diag_missing_copy(out, x, rows, hidden, wait_limit_ns, stream)


def ltxk_status_string(status: int) -> str:
    return _lib.ltxk_status_string(status).decode()


def ltxk_last_cuda_error() -> int:
    return _lib.ltxk_last_cuda_error()


def ltxk_plan_launch(op, rows, hidden, head_dim, mode, vector_ok):
    """Returns (status, Plan)."""
    p = Plan()
    st = _lib.ltxk_plan_launch(op, rows, hidden, head_dim, mode,
                               1 if vector_ok else 0, ctypes.byref(p))
    return st, p


# ---- torch marshalling -----------------------------------------------------

def _check(status, where):
    if status != OK:
        raise LtxkError(status, where)


def _stream_handle(tensor, stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(tensor.device)
    return ctypes.c_void_p(stream.cuda_stream)


def _dev_ptr(t, name, dtype):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _dtype_code(t):
    import torch
    codes = {torch.bfloat16: DTYPE_BF16, torch.float16: DTYPE_F16, torch.float32: DTYPE_F32}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype} (bfloat16, float16 or float32)")
    return codes[t.dtype]


def rms_norm(x, weight=None, eps: float = 1e-6, out=None, stream=None):
    """y = x * weight / sqrt(mean(x^2, -1) + eps) over the last axis
    (bfloat16, float16 or float32; weight and out of x's dtype)."""
    import torch
    code = _dtype_code(x)
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    if out is None:
        out = torch.empty_like(x)
    st = ltxk_rms_norm_dt(_dev_ptr(out, "out", x.dtype), _dev_ptr(x, "x", x.dtype),
                          _dev_ptr(weight, "weight", x.dtype),
                          rows, hidden, eps, code, _stream_handle(x, stream))
    _check(st, "ltxk_rms_norm_dt")
    return out


def rms_norm_rope(x, weight, cos, sin, heads: int, head_dim: int,
                  mode: int = ROPE_INTERLEAVED, eps: float = 1e-6,
                  seq_len: int | None = None, out=None, stream=None):
    """RMSNorm over the last axis (heads*head_dim), then RoPE per head.

    ``cos``/``sin`` are fp32 ``[seq_len, head_dim/2]`` with row r of x using
    table row ``r % seq_len`` (``seq_len`` defaults to the tables' length);
    pass ``seq_len=None`` and tables with one row per row of x for per-row
    tables.
    """
    import torch
    code = _dtype_code(x)
    hidden = heads * head_dim
    if x.shape[-1] != hidden:
        raise ValueError("last axis of x must be heads*head_dim")
    rows = x.numel() // hidden
    if out is None:
        out = torch.empty_like(x)
    table_rows = cos.numel() // (head_dim // 2) if seq_len is None else seq_len
    args = (_dev_ptr(out, "out", x.dtype), _dev_ptr(x, "x", x.dtype),
            _dev_ptr(weight, "weight", x.dtype),
            _dev_ptr(cos, "cos", torch.float32), _dev_ptr(sin, "sin", torch.float32),
            rows, heads, head_dim, mode, eps)
    if code != DTYPE_BF16:
        st = ltxk_rms_norm_rope_dt(*args, table_rows, code, _stream_handle(x, stream))
        _check(st, "ltxk_rms_norm_rope_dt")
    elif table_rows == rows and seq_len is None:
        st = ltxk_rms_norm_rope(*args, _stream_handle(x, stream))
        _check(st, "ltxk_rms_norm_rope")
    else:
        st = ltxk_rms_norm_rope_seq(*args, table_rows, _stream_handle(x, stream))
        _check(st, "ltxk_rms_norm_rope_seq")
    return out


def rms_norm_adaln(x, weight, scale, shift, eps: float = 1e-6, rows_per_cond=None,
                   out=None, stream=None):
    """norm(x) * weight * (1 + scale) + shift over the last axis (bf16).

    ``scale``/``shift`` are ``[n_cond, hidden]``; row r of x uses conditioning
    row ``r // rows_per_cond`` (default: rows / n_cond, e.g. the sequence
    length for x ``[B, S, hidden]`` and conditioning ``[B, hidden]``).
    """
    import torch
    code = _dtype_code(x)
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    n_cond = scale.numel() // hidden if hidden else 0
    if rows_per_cond is None:
        rows_per_cond = max(1, -(-rows // max(1, n_cond)))
    if out is None:
        out = torch.empty_like(x)
    st = ltxk_rms_norm_adaln_dt(_dev_ptr(out, "out", x.dtype), _dev_ptr(x, "x", x.dtype),
                                _dev_ptr(weight, "weight", x.dtype),
                                _dev_ptr(scale, "scale", x.dtype),
                                _dev_ptr(shift, "shift", x.dtype),
                                rows, hidden, rows_per_cond, eps, code, _stream_handle(x, stream))
    _check(st, "ltxk_rms_norm_adaln_dt")
    return out


def rms_norm_host(x, weight=None, eps: float = 1e-6, out=None, staging=None,
                  streams=None):
    """RMSNorm of a HOST tensor ``x`` (bf16, ideally pinned) into a host
    tensor, pipelined over ``streams`` (default: three new streams on the
    current device) and a device ``staging`` buffer (default: 3 x 16 MiB).
    Waits for the result before returning."""
    import torch
    if x.is_cuda:
        raise TypeError("x must be a host tensor (use rms_norm for device tensors)")
    if x.dtype != torch.bfloat16 or not x.is_contiguous():
        raise TypeError("x must be a contiguous bfloat16 tensor")
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    if out is None:
        out = torch.empty_like(x, pin_memory=x.is_pinned())
    dev = torch.device("cuda", torch.cuda.current_device())
    if streams is None:
        streams = [torch.cuda.Stream(dev) for _ in range(3)]
    if staging is None:
        staging = torch.empty(len(streams) * (16 << 20), dtype=torch.uint8, device=dev)
    w = _dev_ptr(weight, "weight", torch.bfloat16)
    st = ltxk_rms_norm_host(out.data_ptr(), x.data_ptr(), w, rows, hidden, eps,
                            staging.data_ptr(), staging.numel() * staging.element_size(),
                            [s.cuda_stream for s in streams], len(streams))
    _check(st, "ltxk_rms_norm_host")
    for s in streams:
        s.synchronize()
    return out


def add_rms_norm(x, residual, weight=None, eps: float = 1e-6, out=None, residual_out=None,
                 stream=None):
    """h = x + residual (bf16), y = RMSNorm(h); returns ``(y, h)``.  Pass
    ``residual_out=residual`` to update the residual stream in place."""
    import torch
    code = _dtype_code(x)
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    if out is None:
        out = torch.empty_like(x)
    if residual_out is None:
        residual_out = torch.empty_like(x)
    st = ltxk_add_rms_norm_dt(_dev_ptr(out, "out", x.dtype),
                              _dev_ptr(residual_out, "residual_out", x.dtype),
                              _dev_ptr(x, "x", x.dtype),
                              _dev_ptr(residual, "residual", x.dtype),
                              _dev_ptr(weight, "weight", x.dtype),
                              rows, hidden, eps, code, _stream_handle(x, stream))
    _check(st, "ltxk_add_rms_norm_dt")
    return out, residual_out


def gelu_tanh(x, out=None, stream=None):
    """Tanh-approximated GELU of a bf16, fp16 or fp32 tensor; ``out=x``
    works in place."""
    import torch
    code = _dtype_code(x)
    if out is None:
        out = torch.empty_like(x)
    if out.shape != x.shape:
        raise ValueError("out must have the shape of x")
    st = ltxk_gelu_tanh_dt(_dev_ptr(out, "out", x.dtype), _dev_ptr(x, "x", x.dtype),
                           x.numel(), code, _stream_handle(x, stream))
    _check(st, "ltxk_gelu_tanh_dt")
    return out


def geglu(x, out=None, stream=None):
    """GEGLU over the last axis: ``x[..., :h] * gelu_tanh(x[..., h:])`` with
    ``h = x.shape[-1] // 2`` (bf16, fp16 or fp32)."""
    import torch
    code = _dtype_code(x)
    if x.shape[-1] % 2:
        raise ValueError("last axis of x must be even")
    hidden = x.shape[-1] // 2
    rows = x.numel() // x.shape[-1] if hidden else 0
    if out is None:
        out = torch.empty(*x.shape[:-1], hidden, dtype=x.dtype, device=x.device)
    st = ltxk_geglu_dt(_dev_ptr(out, "out", x.dtype), _dev_ptr(x, "x", x.dtype),
                       rows, hidden, code, _stream_handle(x, stream))
    _check(st, "ltxk_geglu_dt")
    return out


def rope(x, heads: int, head_dim: int, mode: int = ROPE_INTERLEAVED, grid=None, pairs=None,
         theta: float = 10000.0, out=None, stream=None):
    """Standalone RoPE with angles computed on the device from token
    positions.  ``x``: [..., heads*head_dim] (bfloat16, float16 or float32),
    rows in token order.  ``grid = (T, H, W)`` and ``pairs = (nt, nh, nw)``;
    the default is 1D text over the rows' second-to-last axis: grid
    ``(x.shape[-2] or rows, 1, 1)``, pairs ``(head_dim/2, 0, 0)``."""
    import torch
    code = _dtype_code(x)
    hidden = heads * head_dim
    if x.shape[-1] != hidden:
        raise ValueError("last axis of x must be heads*head_dim")
    rows = x.numel() // hidden if hidden else 0
    if grid is None:
        grid = (x.shape[-2] if x.dim() >= 2 else max(1, rows), 1, 1)
    if pairs is None:
        pairs = (head_dim // 2, 0, 0)
    if out is None:
        out = torch.empty_like(x)
    st = ltxk_rope(_dev_ptr(out, "out", x.dtype), _dev_ptr(x, "x", x.dtype), rows, heads,
                   head_dim, mode, grid[0], grid[1], grid[2], pairs[0], pairs[1], pairs[2],
                   float(theta), code, _stream_handle(x, stream))
    _check(st, "ltxk_rope")
    return out


def rope_tables(head_dim: int, grid, pairs=None, theta: float = 10000.0, tokens=None,
                device=None, stream=None):
    """cos and sin tables ``[tokens, head_dim/2]`` (float32, on the device)
    for ``rms_norm_rope(..., seq_len=tokens)``, with ``rope``'s angles: row s
    is token ``s mod (T*H*W)`` of ``grid = (T, H, W)``; ``pairs`` defaults to
    1D ``(head_dim/2, 0, 0)`` and ``tokens`` to ``T*H*W``."""
    import torch
    T, H, W = grid
    if pairs is None:
        pairs = (head_dim // 2, 0, 0)
    if tokens is None:
        tokens = T * H * W
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    cos = torch.empty(tokens, head_dim // 2, dtype=torch.float32, device=device)
    sin = torch.empty_like(cos)
    st = ltxk_rope_tables(_dev_ptr(cos, "cos", torch.float32), _dev_ptr(sin, "sin", torch.float32),
                          tokens, head_dim, T, H, W, pairs[0], pairs[1], pairs[2], float(theta),
                          _stream_handle(cos, stream))
    _check(st, "ltxk_rope_tables")
    return cos, sin
