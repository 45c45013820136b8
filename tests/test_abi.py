"""Host-side checks of the C ABI: the library loads, exports exactly what
include/ltxk.h declares, rejects bad arguments before any CUDA call, and
plans the kernel the shapes call for.  No GPU work happens here: every call
either fails validation or has rows == 0, and the fake pointers used are
never dereferenced."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ltxk.h")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import rope_element_dit_gb300
    return rope_element_dit_gb300


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"LTXK_API\s+[\w\s\*]+?\b(ltxk_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for required in ("ltxk_rms_norm", "ltxk_rms_norm_rope", "ltxk_rms_norm_rope_seq"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    import ctypes
    lib = ctypes.CDLL(L.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"
    assert sorted(L.EXPORTS) == declared_functions()


def test_exported_symbols_are_only_the_abi(L):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    text_syms = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    ours = {s for s in text_syms if s.startswith("ltxk_")}
    assert ours == set(declared_functions())


# Fake, never-dereferenced device addresses (16-byte aligned, far apart).
A = 0x7F0000000000
B = 0x7F0100000000
W = 0x7F0200000000
C = 0x7F0300000000
S = 0x7F0400000000


def test_status_strings(L):
    for st in range(0, 8):
        assert L.ltxk_status_string(st)
    assert L.ltxk_status_string(99) == "unknown status"


def test_rms_norm_validation(L):
    f = L.ltxk_rms_norm
    assert f(None, B, W, 4, 8, 1e-6, None) == L.ERR_NULL
    assert f(A, None, W, 4, 8, 1e-6, None) == L.ERR_NULL
    assert f(A, B, W, -1, 8, 1e-6, None) == L.ERR_SHAPE
    assert f(A, B, W, 4, 0, 1e-6, None) == L.ERR_SHAPE
    assert f(A, B, W, 4, (1 << 30) + 1, 1e-6, None) == L.ERR_SHAPE
    assert f(A, B, W, 1 << 62, 1 << 10, 1e-6, None) == L.ERR_SHAPE
    assert f(A + 1, B, W, 4, 8, 1e-6, None) == L.ERR_ALIGN
    assert f(A, B + 1, W, 4, 8, 1e-6, None) == L.ERR_ALIGN
    assert f(A, B, W + 1, 4, 8, 1e-6, None) == L.ERR_ALIGN
    # out overlaps x partially (x's rows are 16 bytes, out starts 2 bytes in)
    assert f(A + 2, A, W, 4, 8, 1e-6, None) == L.ERR_OVERLAP
    # out overlaps w
    assert f(A, B, A + 8, 4, 8, 1e-6, None) == L.ERR_OVERLAP
    # rows == 0 is a no-op, also in place; no CUDA call is made
    assert f(A, B, W, 0, 8, 1e-6, None) == L.OK
    assert f(A, A, None, 0, 8, 1e-6, None) == L.OK


def test_rope_validation(L):
    f = L.ltxk_rms_norm_rope
    g = L.ltxk_rms_norm_rope_seq
    assert f(A, B, W, None, S, 4, 2, 8, 0, 1e-6, None) == L.ERR_NULL
    assert f(A, B, W, C, None, 4, 2, 8, 0, 1e-6, None) == L.ERR_NULL
    assert f(A, B, W, C, S, 4, 2, 7, 0, 1e-6, None) == L.ERR_SHAPE      # odd D
    assert f(A, B, W, C, S, 4, 0, 8, 0, 1e-6, None) == L.ERR_SHAPE      # no heads
    assert f(A, B, W, C, S, 4, 2, 0, 0, 1e-6, None) == L.ERR_SHAPE
    assert f(A, B, W, C, S, 4, 1 << 20, 1 << 12, 0, 1e-6, None) == L.ERR_SHAPE
    assert f(A, B, W, C, S, 4, 2, 8, 2, 1e-6, None) == L.ERR_MODE
    assert f(A, B, W, C, S, 4, 2, 8, -1, 1e-6, None) == L.ERR_MODE
    assert f(A, B, W, C + 2, S, 4, 2, 8, 0, 1e-6, None) == L.ERR_ALIGN
    assert f(A, B, W, C, S + 1, 4, 2, 8, 0, 1e-6, None) == L.ERR_ALIGN
    assert g(A, B, W, C, S, 4, 2, 8, 0, 1e-6, 0, None) == L.ERR_SHAPE    # seq_len
    assert g(A, B, W, C, S, 4, 2, 8, 0, 1e-6, -3, None) == L.ERR_SHAPE
    # out overlaps a table: 4 rows x 16 elements x 2 B = 128 B of out
    assert g(A, B, W, A + 64, S, 4, 2, 8, 0, 1e-6, 4, None) == L.ERR_OVERLAP
    assert g(A, B, W, C, A + 100, 4, 2, 8, 1, 1e-6, 4, None) == L.ERR_OVERLAP
    assert g(A, B, W, C, S, 0, 2, 8, 1, 1e-6, 4, None) == L.OK
    assert f(A, A, None, C, S, 0, 2, 8, 1, 1e-6, None) == L.OK


@pytest.mark.parametrize("op,rows,hidden,D,mode,vec,kernel,G,vpl", [
    # plain RMSNorm: rows that split exactly into 3-4 vectors per lane over
    # g >= 4 warps take that split; others the fewest warps per row
    (0, 16384, 2048, 0, 0, True, 1, 1, 8),
    (0, 4096, 2048, 0, 0, True, 1, 1, 8),
    (0, 2048, 2048, 0, 0, True, 1, 2, 4),    # few rows: two warps per row
    (0, 1024, 2048, 0, 0, True, 1, 2, 4),
    (0, 2432, 1536, 0, 0, True, 1, 2, 4),
    (0, 2433, 1536, 0, 0, True, 1, 1, 8),
    (0, 16384, 3072, 0, 0, True, 1, 4, 4),
    (0, 65536, 4096, 0, 0, True, 1, 4, 4),
    (0, 16384, 6144, 0, 0, True, 1, 8, 4),
    (0, 16384, 8192, 0, 0, True, 1, 8, 4),
    (0, 4, 16384, 0, 0, True, 1, 16, 4),
    (0, 4, 32768, 0, 0, True, 1, 32, 4),
    (0, 262143, 2560, 0, 0, True, 1, 1, 12),
    (0, 65536, 5120, 0, 0, True, 1, 2, 12),
    (0, 7, 131072, 0, 0, True, 1, 32, 16),
    (0, 7, 131080, 0, 0, True, 2, 8, 0),     # beyond the register path
    (0, 7, 264, 0, 0, True, 1, 1, 4),
    (0, 7, 4, 0, 0, True, 2, 8, 0),          # hidden % 8 != 0
    (0, 7, 3072, 0, 0, False, 2, 8, 0),      # unaligned pointers
    (3, 4096, 2048, 0, 0, True, 1, 1, 8),    # residual add: 128-thread CTAs
    (2, 4096, 2048, 0, 0, True, 1, 1, 8),    # AdaLN: 256-thread CTAs
    # fused
    (1, 8192, 4096, 128, 0, True, 1, 4, 4),  # fused rows split over 4 warps
    (1, 6144, 2048, 64, 1, True, 1, 1, 8),
    (1, 9, 48, 24, 0, True, 1, 1, 4),
    (1, 9, 48, 24, 1, True, 2, 8, 0),        # split needs head_dim % 16
    (1, 9, 40, 20, 0, True, 2, 8, 0),        # interleaved needs head_dim % 8
    (1, 9, 4096, 128, 1, False, 2, 8, 0),
    (1, 9, 10240, 128, 1, True, 1, 8, 8),
])
def test_plan(L, op, rows, hidden, D, mode, vec, kernel, G, vpl):
    st, p = L.ltxk_plan_launch(op, rows, hidden, D, mode, vec)
    assert st == L.OK
    assert (p.kernel, p.group_warps, p.vec_per_lane) == (kernel, G, vpl)
    if kernel in (L.KERNEL_ROWS_VEC, L.KERNEL_ROWS_TMA):
        # the slots cover the row exactly once
        nv = hidden // 8
        assert 32 * G * vpl >= nv
    if kernel == L.KERNEL_ROWS_VEC:
        # plain and AdaLN rows of one or two warps run eight or four rows per
        # 256-thread CTA, the others 128 threads (or one row group)
        row_only = op in (L.OP_RMS_NORM, L.OP_RMS_NORM_ADALN)
        assert p.block_threads == (256 if row_only and G <= 2 else max(128, 32 * G))
        assert p.rows_per_cta == p.block_threads // (32 * G)
        # AdaLN's 16-bit rows stage the CTA's conditioning row (scale, shift)
        assert p.stages == 0
        assert p.smem_bytes == (4 * hidden if op == L.OP_RMS_NORM_ADALN else 0)
    if kernel == L.KERNEL_ROWS_TMA:
        stride = (hidden * 2 + 127) // 128 * 128
        assert p.block_threads == 256 and p.rows_per_cta == 8
        assert 1 <= p.stages <= 8
        assert p.smem_bytes == 512 + 8 * p.stages * stride
        assert p.smem_bytes <= 227 * 1024


def test_plan_follows_path_setting(L):
    try:
        assert L.ltxk_set_path(L.PATH_REGISTERS) == L.PATH_AUTO
        st, p = L.ltxk_plan_launch(0, 16384, 2560, 0, 0, True)
        assert (p.kernel, p.group_warps, p.vec_per_lane) == (L.KERNEL_ROWS_VEC, 1, 12)
        assert L.ltxk_set_path(L.PATH_TMA) == L.PATH_REGISTERS
        st, p = L.ltxk_plan_launch(0, 16384, 2560, 0, 0, True)
        assert p.kernel == L.KERNEL_ROWS_TMA
        assert p.stages >= 1 and p.smem_bytes > 0
        # beyond one warp per row the register kernel stays
        st, p = L.ltxk_plan_launch(0, 16384, 5120, 0, 0, True)
        assert p.kernel == L.KERNEL_ROWS_VEC
        assert L.ltxk_set_path(9) == -1
    finally:
        L.ltxk_set_path(L.PATH_AUTO)


def test_diag_validation(L):
    f = L.ltxk_diag_missing_copy
    assert f(None, B, 4, 8, 10**6, None) == L.ERR_NULL
    assert f(A, B, 4, 4100, 10**6, None) == L.ERR_SHAPE      # hidden > 4096
    assert f(A, B, 4, 12, 10**6, None) == L.ERR_SHAPE        # hidden % 8
    assert f(A, B, 4, 8, 10, None) == L.ERR_SHAPE            # limit too short
    assert f(A, B, 4, 8, 10**11, None) == L.ERR_SHAPE        # limit too long
    assert f(A + 2, B, 4, 8, 10**6, None) == L.ERR_ALIGN
    assert f(A, B, 0, 8, 10**6, None) == L.OK


def test_plan_rows_zero_and_errors(L):
    st, p = L.ltxk_plan_launch(0, 0, 4096, 0, 0, True)
    assert st == L.OK and p.kernel == L.KERNEL_NONE
    assert L.ltxk_plan_launch(1, 4, 4096, 7, 0, True)[0] == L.ERR_SHAPE
    assert L.ltxk_plan_launch(1, 4, 4096, 128, 5, True)[0] == L.ERR_MODE
    assert L.ltxk_plan_launch(7, 4, 4096, 128, 0, True)[0] == L.ERR_MODE


def test_product_and_oracle_share_nothing():
    """Neither side imports the other; they share no source file."""
    pkg = os.path.join(ROOT, "rope_element_dit_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"\boracle\b", text), f"{fn} names the oracle"
                assert "synth" not in text, f"{fn} uses the input generator"
    for fn in os.listdir(os.path.join(ROOT, "oracle")):
        if fn.endswith((".py", ".c")):
            text = open(os.path.join(ROOT, "oracle", fn)).read()
            assert "rope_element_dit_gb300" not in text and "ltxk" not in text, fn


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    """Importing the binding with no built library raises ImportError (no
    silent fallback)."""
    import importlib.util
    import shutil
    d = tmp_path / "pkgcopy"
    d.mkdir()
    shutil.copy(os.path.join(ROOT, "rope_element_dit_gb300", "__init__.py"), d / "__init__.py")
    spec = importlib.util.spec_from_file_location("pkgcopy", d / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)


def test_adaln_validation(L):
    f = L.ltxk_rms_norm_adaln
    assert f(A, B, W, None, S, 4, 8, 2, 1e-6, None) == L.ERR_NULL
    assert f(A, B, W, C, None, 4, 8, 2, 1e-6, None) == L.ERR_NULL
    assert f(A, B, W, C, S, 4, 8, 0, 1e-6, None) == L.ERR_SHAPE        # rows_per_cond
    assert f(A, B, W, C + 1, S, 4, 8, 2, 1e-6, None) == L.ERR_ALIGN
    # out (4 rows x 8 x 2 B = 64 B) overlaps the scale
    assert f(A, B, W, A + 32, S, 4, 8, 2, 1e-6, None) == L.ERR_OVERLAP
    assert f(A, B, W, C, A, 4, 8, 2, 1e-6, None) == L.ERR_OVERLAP
    assert f(A, B, W, C, S, 0, 8, 2, 1e-6, None) == L.OK


def test_adaln_plan(L):
    st, p = L.ltxk_plan_launch(L.OP_RMS_NORM_ADALN, 12288, 2048, 0, 0, True)
    assert st == L.OK and (p.kernel, p.group_warps, p.vec_per_lane) == (1, 1, 8)
    # 16-bit rows stage the CTA's conditioning row (scale, shift) in shared
    # memory, up to hidden 12288 (48 KB, no opt-in); fp32 rows do not
    assert p.smem_bytes == 4 * 2048
    st, p = L.ltxk_plan_launch(L.OP_RMS_NORM_ADALN, 12288, 3072, 0, 0, True)
    assert (p.kernel, p.group_warps, p.vec_per_lane) == (1, 4, 4) and p.smem_bytes == 4 * 3072
    st, p = L.ltxk_plan_launch_dt(L.OP_RMS_NORM_ADALN, L.DTYPE_F32, 12288, 2048, 0, 0, True)
    assert p.kernel == L.KERNEL_ROWS_VEC and p.smem_bytes == 0
    st, p = L.ltxk_plan_launch(L.OP_RMS_NORM_ADALN, 8, 16384, 0, 0, True)
    assert p.kernel == L.KERNEL_ROWS_VEC and p.smem_bytes == 0
    st, p = L.ltxk_plan_launch(L.OP_RMS_NORM_ADALN, 12288, 3072, 0, 0, False)
    assert p.kernel == L.KERNEL_ROWS_ELEM
    try:   # the TMA ring has no AdaLN form: the register kernel stays
        L.ltxk_set_path(L.PATH_TMA)
        st, p = L.ltxk_plan_launch(L.OP_RMS_NORM_ADALN, 12288, 2048, 0, 0, True)
        assert p.kernel == L.KERNEL_ROWS_VEC
    finally:
        L.ltxk_set_path(L.PATH_AUTO)


def test_host_pipeline_validation(L):
    f = L.ltxk_rms_norm_host
    st = [0, 0]
    assert f(None, B, W, 4, 8, 1e-6, C, 1 << 20, st, 2) == L.ERR_NULL
    assert f(A, B, W, 4, 8, 1e-6, None, 1 << 20, st, 2) == L.ERR_NULL
    assert f(A, B, W, 4, 8, 1e-6, C, 1 << 20, st, 0) == L.ERR_SHAPE       # no stream
    assert f(A, B, W, 4, 8, 1e-6, C, 1 << 20, st * 5, 10) == L.ERR_SHAPE  # too many
    assert f(A, B, W, 4, 8, 1e-6, C, 16, st, 2) == L.ERR_SHAPE            # < 1 row/slot
    assert f(A, B, W, 4, 8, 1e-6, C + 16, 1 << 20, st, 2) == L.ERR_ALIGN  # staging 256 B
    assert f(A + 1, B, W, 4, 8, 1e-6, C, 1 << 20, st, 2) == L.ERR_ALIGN
    assert f(A, B, C + 64, 4, 8, 1e-6, C, 1 << 20, st, 2) == L.ERR_OVERLAP  # w in staging
    assert f(A, B, W, 0, 8, 1e-6, C, 1 << 20, st, 2) == L.OK


def test_add_norm_validation(L):
    f = L.ltxk_add_rms_norm
    D = 0x7F0500000000
    E = 0x7F0600000000
    assert f(A, None, B, C, W, 4, 8, 1e-6, None) == L.ERR_NULL
    assert f(A, D, B, None, W, 4, 8, 1e-6, None) == L.ERR_NULL
    assert f(A, D + 1, B, C, W, 4, 8, 1e-6, None) == L.ERR_ALIGN
    assert f(A, A + 16, B, C, W, 4, 8, 1e-6, None) == L.ERR_OVERLAP      # outputs overlap
    assert f(A, D, B, D + 2, W, 4, 8, 1e-6, None) == L.ERR_OVERLAP       # partial alias
    # exact aliases are allowed (rows == 0: nothing is launched)
    assert f(A, D, A, D, W, 0, 8, 1e-6, None) == L.OK
    assert f(A, D, E, C, D + 8, 4, 8, 1e-6, None) == L.ERR_OVERLAP       # w in residual_out
    st, p = L.ltxk_plan_launch(L.OP_ADD_RMS_NORM, 16384, 3072, 0, 0, True)
    assert st == L.OK and (p.kernel, p.group_warps, p.vec_per_lane) == (1, 4, 4)


def test_gelu_validation(L):
    """Argument errors come back before any CUDA call (fake addresses are
    never dereferenced; n == 0 launches nothing)."""
    g = L.ltxk_gelu_tanh
    assert g(None, B, 16, None) == L.ERR_NULL
    assert g(A, None, 16, None) == L.ERR_NULL
    assert g(A, B, -1, None) == L.ERR_SHAPE
    assert g(A, B, (1 << 40) + 1, None) == L.ERR_SHAPE
    assert g(A + 1, B, 16, None) == L.ERR_ALIGN
    assert g(A, B + 1, 16, None) == L.ERR_ALIGN
    assert g(A, A + 2, 16, None) == L.ERR_OVERLAP
    assert g(A + 30, A, 16, None) == L.ERR_OVERLAP
    assert g(A, A, 0, None) == L.OK                       # in place, empty
    assert g(A, B, 0, None) == L.OK


def test_geglu_validation(L):
    f = L.ltxk_geglu
    assert f(None, B, 4, 8, None) == L.ERR_NULL
    assert f(A, None, 4, 8, None) == L.ERR_NULL
    assert f(A, B, -1, 8, None) == L.ERR_SHAPE
    assert f(A, B, 4, 0, None) == L.ERR_SHAPE
    assert f(A, B, 4, (1 << 30) + 1, None) == L.ERR_SHAPE
    assert f(A, B, (1 << 31) + 1, 1 << 9, None) == L.ERR_SHAPE  # rows * hidden > 2^40
    assert f(A + 1, B, 4, 8, None) == L.ERR_ALIGN
    assert f(A, B + 3, 4, 8, None) == L.ERR_ALIGN
    assert f(A, A, 4, 8, None) == L.ERR_OVERLAP          # out inside x: never in place
    assert f(A + 120, A, 4, 8, None) == L.ERR_OVERLAP    # last bytes of x
    assert f(A, B, 0, 8, None) == L.OK


def test_gelu_geglu_dtype_validation(L):
    """The per-format entry points: unknown dtypes, the element size's
    alignment and byte extents, all before any CUDA call."""
    g, f = L.ltxk_gelu_tanh_dt, L.ltxk_geglu_dt
    assert g(A, B, 16, 3, None) == L.ERR_DTYPE
    assert g(None, B, 16, -1, None) == L.ERR_DTYPE         # dtype checked first
    assert f(A, B, 4, 8, 5, None) == L.ERR_DTYPE
    assert g(A + 2, B, 16, L.DTYPE_F32, None) == L.ERR_ALIGN    # fp32 wants 4 bytes
    assert g(A + 1, B, 16, L.DTYPE_F16, None) == L.ERR_ALIGN
    assert f(A, B + 2, 4, 8, L.DTYPE_F32, None) == L.ERR_ALIGN
    assert g(A + 60, A, 16, L.DTYPE_F32, None) == L.ERR_OVERLAP  # 64 bytes of fp32
    assert g(A + 30, A, 16, L.DTYPE_F16, None) == L.ERR_OVERLAP
    assert f(A + 248, A, 4, 8, L.DTYPE_F32, None) == L.ERR_OVERLAP   # x is 256 bytes
    assert f(A + 256, A, 0, 8, L.DTYPE_F32, None) == L.OK
    for dt in (L.DTYPE_BF16, L.DTYPE_F16, L.DTYPE_F32):
        assert g(A, A, 0, dt, None) == L.OK and f(A, B, 0, 8, dt, None) == L.OK
        assert g(A, B, -1, dt, None) == L.ERR_SHAPE and f(A, B, 4, 0, dt, None) == L.ERR_SHAPE


def test_plans_per_format(L):
    """fp32 rows use at most 8 slots per lane; the TMA ring stays bf16-only."""
    old = L.ltxk_set_path(L.PATH_TMA)
    try:
        for op in (L.OP_RMS_NORM, L.OP_RMS_NORM_ROPE):
            st, p = L.ltxk_plan_launch_dt(op, L.DTYPE_F16, 64, 2048, 64, 1, True)
            assert st == L.OK and p.kernel == L.KERNEL_ROWS_VEC
        st, p = L.ltxk_plan_launch_dt(L.OP_RMS_NORM, L.DTYPE_BF16, 64, 2048, 0, 0, True)
        assert st == L.OK and p.kernel == L.KERNEL_ROWS_TMA
    finally:
        L.ltxk_set_path(old)
    st, p = L.ltxk_plan_launch_dt(L.OP_RMS_NORM, L.DTYPE_F32, 64, 4096 * 3, 0, 0, True)
    assert st == L.OK and p.vec_per_lane <= 8


def test_dtype_validation(L):
    """Unknown dtypes and element-size rules come back before any CUDA call."""
    assert L.ltxk_rms_norm_dt(A, B, W, 4, 8, 1e-6, 3, None) == L.ERR_DTYPE
    assert L.ltxk_rms_norm_dt(None, B, W, 4, 8, 1e-6, -1, None) == L.ERR_DTYPE
    assert L.ltxk_rms_norm_rope_dt(A, B, W, C, C, 4, 2, 8, 0, 1e-6, 4, 7, None) == L.ERR_DTYPE
    assert L.ltxk_rms_norm_adaln_dt(A, B, W, C, C, 4, 8, 2, 1e-6, 9, None) == L.ERR_DTYPE
    assert L.ltxk_add_rms_norm_dt(A, C, B, W, None, 4, 8, 1e-6, 5, None) == L.ERR_DTYPE
    st, _ = L.ltxk_plan_launch_dt(L.OP_RMS_NORM, 3, 4, 8, 0, 0, True)
    assert st == L.ERR_DTYPE
    # fp32 elements need 4-byte alignment; 2 bytes is enough for the 16-bit types
    assert L.ltxk_rms_norm_dt(A, B + 2, W, 4, 8, 1e-6, L.DTYPE_F32, None) == L.ERR_ALIGN
    assert L.ltxk_rms_norm_dt(A, B + 2, W, 0, 8, 1e-6, L.DTYPE_F16, None) == L.OK
    # overlap is measured in bytes of the element type: 4 x 8 fp32 = 128 bytes
    assert L.ltxk_rms_norm_dt(A, A + 96, None, 4, 8, 1e-6, L.DTYPE_F32, None) == L.ERR_OVERLAP
    assert L.ltxk_rms_norm_dt(A, A + 64, None, 0, 8, 1e-6, L.DTYPE_F16, None) == L.OK
    assert L.ltxk_rms_norm_dt(A, B, A + 100, 4, 8, 1e-6, L.DTYPE_F32, None) == L.ERR_OVERLAP
    assert L.ltxk_add_rms_norm_dt(A, A + 64, B, C, None, 4, 8, 1e-6, L.DTYPE_F32,
                                  None) == L.ERR_OVERLAP
    assert L.ltxk_rms_norm_adaln_dt(A, B, None, A + 124, C, 4, 8, 2, 1e-6, L.DTYPE_F32,
                                    None) == L.ERR_OVERLAP
    assert L.ltxk_status_string(L.ERR_DTYPE) == "unknown element type"


def test_rope_validation(L):
    """Standalone RoPE: argument errors come back before any CUDA call."""
    f = L.ltxk_rope
    ok = dict(rows=4, heads=2, head_dim=8, mode=0, g=(4, 1, 1), p=(4, 0, 0), theta=1e4,
              dtype=L.DTYPE_BF16)

    def call(out=A, x=B, **kw):
        a = dict(ok, **kw)
        return f(out, x, a["rows"], a["heads"], a["head_dim"], a["mode"], *a["g"], *a["p"],
                 a["theta"], a["dtype"], None)

    assert call(dtype=7) == L.ERR_DTYPE
    assert call(out=None) == L.ERR_NULL and call(x=None) == L.ERR_NULL
    assert call(mode=2) == L.ERR_MODE
    assert call(rows=-1) == L.ERR_SHAPE
    assert call(head_dim=7, p=(3, 0, 0)) == L.ERR_SHAPE
    assert call(head_dim=1024, p=(512, 0, 0)) == L.ERR_SHAPE         # over 512
    assert call(p=(3, 0, 0)) == L.ERR_SHAPE                          # pairs must add up
    assert call(p=(5, -1, 0)) == L.ERR_SHAPE
    assert call(g=(0, 1, 1)) == L.ERR_SHAPE
    assert call(theta=0.0) == L.ERR_SHAPE and call(theta=float("nan")) == L.ERR_SHAPE
    assert call(x=B + 1) == L.ERR_ALIGN
    assert call(x=B + 2, dtype=L.DTYPE_F32) == L.ERR_ALIGN
    assert call(out=A, x=A + 16) == L.ERR_OVERLAP
    assert call(rows=0) == L.OK                                       # nothing launched
    assert call(rows=0, out=A, x=A) == L.OK


def test_host_pipeline_rejects_partial_overlap(L):
    f = L.ltxk_rms_norm_host
    S = 0x7F0800000000
    # 4 rows x 8 bf16 = 64 bytes: out 16 bytes into x
    assert f(A + 16, A, None, 4, 8, 1e-6, S, 1 << 20, [0], 1) == L.ERR_OVERLAP
    assert f(A, A + 62, None, 4, 8, 1e-6, S, 1 << 20, [0], 1) == L.ERR_OVERLAP
    assert f(A, A, None, 0, 8, 1e-6, S, 1 << 20, [0], 1) == L.OK      # in place, empty


def test_helpers_reject_host_tensors(L):
    """The torch helpers take device tensors only: a host tensor is an error
    before any CUDA call, never a CPU computation."""
    import torch
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    cos = torch.zeros(4, 8)
    for call in (lambda: L.rms_norm(x),
                 lambda: L.rms_norm_rope(x, None, cos, cos, 4, 16, L.ROPE_INTERLEAVED, 1e-6),
                 lambda: L.rms_norm_adaln(x, None, x[:1], x[:1]),
                 lambda: L.add_rms_norm(x, x),
                 lambda: L.gelu_tanh(x),
                 lambda: L.geglu(x),
                 lambda: L.rope(x, 4, 16, L.ROPE_INTERLEAVED)):
        with pytest.raises(TypeError):
            call()
    with pytest.raises(TypeError):
        L.rms_norm(torch.zeros(4, 64, dtype=torch.float64))


def test_rope_tables_validation(L):
    f = L.ltxk_rope_tables
    args = (4096, 128, 4096, 1, 1, 64, 0, 0, 10000.0, None)
    assert f(None, B, *args) == L.ERR_NULL
    assert f(A, None, *args) == L.ERR_NULL
    assert f(A, B, -1, 128, 4096, 1, 1, 64, 0, 0, 1e4, None) == L.ERR_SHAPE
    assert f(A, B, 16, 127, 16, 1, 1, 63, 0, 0, 1e4, None) == L.ERR_SHAPE      # odd head_dim
    assert f(A, B, 16, 1026, 16, 1, 1, 513, 0, 0, 1e4, None) == L.ERR_SHAPE    # > 256 pairs
    assert f(A, B, 16, 128, 16, 1, 1, 63, 0, 0, 1e4, None) == L.ERR_SHAPE      # pairs != D/2
    assert f(A, B, 16, 128, 0, 1, 1, 64, 0, 0, 1e4, None) == L.ERR_SHAPE       # empty grid
    assert f(A, B, 16, 128, 16, 1, 1, 64, 0, 0, -1.0, None) == L.ERR_SHAPE     # theta <= 0
    assert f(A + 2, B, 16, 128, 16, 1, 1, 64, 0, 0, 1e4, None) == L.ERR_ALIGN
    assert f(A, A + 64, 16, 128, 16, 1, 1, 64, 0, 0, 1e4, None) == L.ERR_OVERLAP  # 16 x 64 x 4 B
    assert f(A, B, 0, 128, 16, 1, 1, 64, 0, 0, 1e4, None) == L.OK              # no tokens


# The launch each bench workload shape gets: (kernel, warps per row, slots per
# lane, threads per CTA, rows per CTA, dynamic shared memory).  The committed
# ncu figures (launch lists, captures, DRAM traffic per kernel instance) were
# taken on these launches; a planner change that moves a shape to another
# instance or CTA shape has to be measured again.
BENCH_PLANS = [
    ("rms_norm_1x1024x2048", (1, 2, 4, 256, 4, 0)),
    ("rms_norm_2x1024x2048", (1, 2, 4, 256, 4, 0)),
    ("rms_norm_4x1024x2048", (1, 1, 8, 256, 8, 0)),
    ("rms_norm_2x4096x3072", (1, 4, 4, 128, 1, 0)),
    ("rms_norm_4x4096x3072", (1, 4, 4, 128, 1, 0)),
    ("rms_norm_rope_interleaved_2x4096x32x128", (1, 4, 4, 128, 1, 0)),
    ("rms_norm_split_rope_1x6144x32x64", (1, 1, 8, 128, 4, 0)),
    ("rms_norm_4x16384x4096", (1, 4, 4, 128, 1, 0)),
    ("rms_norm_262143x2560", (1, 1, 12, 256, 8, 0)),
    ("rms_norm_65536x5120", (1, 2, 12, 256, 4, 0)),
    ("rms_norm_adaln_2x6144x2048", (1, 1, 8, 256, 8, 8192)),
    ("add_rms_norm_4x4096x3072", (1, 4, 4, 128, 1, 0)),
    ("rms_norm_f16_4x4096x3072", (1, 4, 4, 128, 1, 0)),
    ("rms_norm_f32_4x4096x3072", (1, 4, 4, 128, 1, 0)),
]


@pytest.mark.parametrize("name,plan", BENCH_PLANS)
def test_bench_workload_plans(L, name, plan):
    import sys
    sys.path.insert(0, ROOT)
    import synth
    case = {c.name: c for w in synth.WORKLOADS.values() for c in w}[name]
    op = {"norm": L.OP_RMS_NORM, "rope": L.OP_RMS_NORM_ROPE, "adaln": L.OP_RMS_NORM_ADALN,
          "add_norm": L.OP_ADD_RMS_NORM}[case.kind]
    dt = {"bf16": L.DTYPE_BF16, "f16": L.DTYPE_F16, "f32": L.DTYPE_F32}[case.dtype]
    st, p = L.ltxk_plan_launch_dt(op, dt, case.rows, case.hidden, case.head_dim or 0,
                                  case.mode or 0, True)
    assert st == L.OK
    assert (p.kernel, p.group_warps, p.vec_per_lane, p.block_threads, p.rows_per_cta,
            p.smem_bytes) == plan
