"""GPU parity of the row operations in the pages' other two precision modes
("cuda-kernels" page, "Supported Data Types": __half and float besides
__nv_bfloat16) against the fp64 oracle, through the *_dt entry points.

fp16 rows: x * w is exact in fp32 (11-bit significands), so, as for bf16,
every element must be within 1 fp16 ulp of the oracle's correctly rounded
value (AdaLN: the bf16 AdaLN rule, because the shift can cancel).

fp32 rows: x * w rounds, and the output's own rounding is as fine as the
kernel's fp32 error, so the tolerance is the bound derived from the
arithmetic: delta(H) = (H/128 + 26) 2^-24 for the sum of squares, the mean,
eps and rsqrtf (the chain of the bf16 AdaLN bound), plus a few roundings of
the products; for RoPE the rotation error scales with the pair's inputs,
not with the possibly cancelled output.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import rope_element_dit_gb300 as L
import synth
from oracle.compare import compare_fmt, compare_fmt_bounded

pytestmark = pytest.mark.gpu

THREADS = min(32, os.cpu_count() or 1)
GUARD = 64
FMTS = {"f16": (np.float16, torch.float16, L.DTYPE_F16, np.uint16, 0x7E01),
        "f32": (np.float32, torch.float32, L.DTYPE_F32, np.uint32, 0x7FC00001)}
U = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU parity tests need a CUDA device"
    torch.cuda.set_device(0)
    assert torch.cuda.get_device_capability(0) == (10, 3)


def stream():
    return torch.cuda.current_stream().cuda_stream


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def guarded(n, fmt):
    """Device buffer of n elements with GUARD canary elements on each side."""
    _, tt, _, ut, canary = FMTS[fmt]   # both canaries are NaNs below 2^15 / 2^31
    it = torch.int16 if ut == np.uint16 else torch.int32
    whole = torch.full((n + 2 * GUARD,), canary, dtype=it, device="cuda")
    return whole, whole[GUARD:GUARD + n].view(tt)


def check_guard(whole, n, fmt):
    ut, canary = FMTS[fmt][3], FMTS[fmt][4]
    h = whole.cpu().numpy().view(ut)
    assert np.all(h[:GUARD] == canary) and np.all(h[GUARD + n:] == canary), \
        "kernel wrote outside its output"


def host(t, fmt):
    return t.cpu().numpy().astype(FMTS[fmt][0], copy=False).reshape(-1)


def delta(H):
    return (H / 128 + 26) * U


def check_plain(got, x, w, eps, fmt, what):
    y, ye = oracle.rms_norm(x, w, eps, exact=True, threads=THREADS)
    if fmt == "f16":
        r = compare_fmt(got, y.reshape(-1))
    else:
        r = compare_fmt_bounded(got, ye, (delta(x.shape[-1]) + 4 * U) * np.abs(ye.reshape(-1)))
    assert r["ok"], f"{what}: {r}"


def pair_magnitude(n, head_dim, mode):
    """|n_a| + |n_b| for the rotation pair of every element."""
    rows, H = n.shape
    a = np.abs(n).reshape(rows, H // head_dim, head_dim)
    if mode == 0:
        m = a.reshape(rows, H // head_dim, head_dim // 2, 2).sum(-1, keepdims=True)
        m = np.broadcast_to(m, a.reshape(rows, H // head_dim, head_dim // 2, 2).shape)
    else:
        P = head_dim // 2
        s = a[..., :P] + a[..., P:]
        m = np.concatenate([s, s], axis=-1)
    return np.asarray(m).reshape(rows, H)


def check_rope(got, x, w, c, s, heads, D, mode, eps, seq_len, fmt, what):
    y, ye = oracle.rms_norm_rope(x, w, c, s, heads, D, mode, eps, table_rows=seq_len,
                                 exact=True, threads=THREADS)
    if fmt == "f16":
        r = compare_fmt(got, y.reshape(-1))
    else:
        _, n = oracle.rms_norm(x, w, eps, exact=True, threads=THREADS)
        bound = delta(heads * D) * np.abs(ye) + 8 * U * pair_magnitude(n, D, mode)
        r = compare_fmt_bounded(got, ye, bound)
    assert r["ok"], f"{what}: {r}"


def adaln_bound(H, y_exact, shift_rows):
    d = delta(H)
    ns = np.abs(y_exact - shift_rows)
    return 2 * d * ns + 2.0 ** -22 * (ns + np.abs(shift_rows))


# ------------------------------------------------------------------ RMSNorm --

SHAPES = [(1, 4), (37, 24), (9, 40), (1000, 264), (17, 2056), (1001, 3072), (33, 5120),
          (19, 8200), (3, 65536), (2, 65544), (2049, 2048), (5, 7), (9, 4096), (5, 8192),
          (3, 16384), (2, 32768)]


@pytest.mark.parametrize("fmt", ["f16", "f32"])
@pytest.mark.parametrize("rows,hidden", SHAPES)
@pytest.mark.parametrize("with_w", [True, False])
def test_rms_norm_shapes(fmt, rows, hidden, with_w):
    seed = 4000 + rows + hidden
    x = synth.normal_with_outliers_bf16(seed, rows * hidden, 0.01, 50.0, fmt=fmt)
    x = x.reshape(rows, hidden)
    w = synth.normal_bf16(seed, 2, hidden, 1.0, 0.1, fmt=fmt) if with_w else None
    whole, out = guarded(rows * hidden, fmt)
    xd, wd = dev(x), (None if w is None else dev(w))
    st = L.ltxk_rms_norm_dt(out.data_ptr(), xd.data_ptr(), None if wd is None else wd.data_ptr(),
                            rows, hidden, 1e-6, FMTS[fmt][2], stream())
    assert st == L.OK, L.ltxk_status_string(st)
    torch.cuda.synchronize()
    check_guard(whole, rows * hidden, fmt)
    check_plain(host(out, fmt), x, w, 1e-6, fmt, f"{fmt} {rows}x{hidden}")


@pytest.mark.parametrize("fmt", ["f16", "f32"])
def test_workload_full_size(fmt):
    case = synth.WORKLOADS[fmt][0]
    inp = synth.make_inputs(case)
    x, w = inp["x"], inp["w"]
    n = case.rows * case.hidden
    whole, out = guarded(n, fmt)
    xd, wd = dev(x), dev(w)
    st = L.ltxk_rms_norm_dt(out.data_ptr(), xd.data_ptr(), wd.data_ptr(), case.rows,
                            case.hidden, case.eps, FMTS[fmt][2], stream())
    assert st == L.OK
    torch.cuda.synchronize()
    check_guard(whole, n, fmt)
    check_plain(host(out, fmt), x, w, case.eps, fmt, case.name)


@pytest.mark.parametrize("fmt", ["f16", "f32"])
def test_unaligned_and_in_place(fmt):
    rows, hidden = 37, 3072
    x = synth.normal_bf16(71, 0, rows * hidden, fmt=fmt).reshape(rows, hidden)
    w = synth.normal_bf16(71, 2, hidden, 1.0, 0.1, fmt=fmt)
    pad = np.zeros(1, x.dtype)
    xb, wb = dev(np.concatenate([pad, x.ravel()])), dev(np.concatenate([pad, w]))
    whole, out = guarded(rows * hidden + 1, fmt)
    st = L.ltxk_rms_norm_dt(out[1:].data_ptr(), xb[1:].data_ptr(), wb[1:].data_ptr(), rows,
                            hidden, 1e-6, FMTS[fmt][2], stream())
    assert st == L.OK
    torch.cuda.synchronize()
    check_guard(whole, rows * hidden + 1, fmt)
    check_plain(host(out[1:], fmt), x, w, 1e-6, fmt, "unaligned")
    xd, wd = dev(x), dev(w)
    st = L.ltxk_rms_norm_dt(xd.data_ptr(), xd.data_ptr(), wd.data_ptr(), rows, hidden, 1e-6,
                            FMTS[fmt][2], stream())
    assert st == L.OK
    torch.cuda.synchronize()
    check_plain(host(xd, fmt), x, w, 1e-6, fmt, "in place")


def test_f16_overflow_to_infinity():
    """Outputs beyond 65504 round to infinity on both sides."""
    rows, hidden = 8, 1024
    x = synth.normal_bf16(72, 0, rows * hidden, fmt="f16").reshape(rows, hidden)
    w = np.full(hidden, 30000.0, np.float16)
    out = torch.empty(rows * hidden, dtype=torch.float16, device="cuda")
    xd, wd = dev(x), dev(w)
    assert L.ltxk_rms_norm_dt(out.data_ptr(), xd.data_ptr(), wd.data_ptr(), rows, hidden, 1e-6,
                              L.DTYPE_F16, stream()) == L.OK
    torch.cuda.synchronize()
    got = host(out, "f16")
    assert np.isinf(got).sum() > 100
    check_plain(got, x, w, 1e-6, "f16", "overflow")


# --------------------------------------------------------------------- RoPE --

# (5003, 8, 64, 61): more rows than one pass of the persistent grid, so the
# warps of the software-pipelined split-half kernel carry their next row
ROPE = [(64, 32, 128, 64), (48, 32, 64, 16), (33, 4, 128, 7), (21, 3, 16, 5), (9, 2, 6, 4),
        (7, 5, 24, 3), (5003, 8, 64, 61)]


@pytest.mark.parametrize("fmt", ["f16", "f32"])
@pytest.mark.parametrize("rows,heads,D,seq_len", ROPE)
@pytest.mark.parametrize("mode", [0, 1])
def test_rope(fmt, rows, heads, D, seq_len, mode):
    H = heads * D
    seed = 5000 + rows + H + mode
    x = synth.normal_bf16(seed, 0, rows * H, fmt=fmt).reshape(rows, H)
    w = synth.normal_bf16(seed, 2, H, 1.0, 0.1, fmt=fmt)
    c, s = synth.rope_table_1d(seq_len, D)
    whole, out = guarded(rows * H, fmt)
    xd, wd, cd, sd = dev(x), dev(w), dev(c), dev(s)
    st = L.ltxk_rms_norm_rope_dt(out.data_ptr(), xd.data_ptr(), wd.data_ptr(), cd.data_ptr(),
                                 sd.data_ptr(), rows, heads, D, mode, 1e-6, seq_len,
                                 FMTS[fmt][2], stream())
    assert st == L.OK, L.ltxk_status_string(st)
    torch.cuda.synchronize()
    check_guard(whole, rows * H, fmt)
    check_rope(host(out, fmt), x, w, c, s, heads, D, mode, 1e-6, seq_len, fmt,
               f"{fmt} mode {mode} {rows}x{heads}x{D}")


# -------------------------------------------------------------------- AdaLN --

@pytest.mark.parametrize("fmt", ["f16", "f32"])
@pytest.mark.parametrize("rows,hidden,rpc,with_w", [(96, 2048, 48, False), (37, 3072, 10, True),
                                                    (9, 40, 4, True), (5, 7, 2, False)])
def test_adaln(fmt, rows, hidden, rpc, with_w):
    seed = 6000 + rows + hidden
    x = synth.normal_bf16(seed, 0, rows * hidden, fmt=fmt).reshape(rows, hidden)
    w = synth.normal_bf16(seed, 2, hidden, 1.0, 0.1, fmt=fmt) if with_w else None
    n_cond = -(-rows // rpc)
    sc = synth.normal_bf16(seed, 3, n_cond * hidden, 0.0, 0.5, fmt=fmt).reshape(n_cond, hidden)
    sh = synth.normal_bf16(seed, 4, n_cond * hidden, 0.0, 0.5, fmt=fmt).reshape(n_cond, hidden)
    whole, out = guarded(rows * hidden, fmt)
    xd, scd, shd = dev(x), dev(sc), dev(sh)
    wd = None if w is None else dev(w)
    st = L.ltxk_rms_norm_adaln_dt(out.data_ptr(), xd.data_ptr(),
                                  None if wd is None else wd.data_ptr(), scd.data_ptr(),
                                  shd.data_ptr(), rows, hidden, rpc, 1e-6, FMTS[fmt][2], stream())
    assert st == L.OK, L.ltxk_status_string(st)
    torch.cuda.synchronize()
    check_guard(whole, rows * hidden, fmt)
    _, ye = oracle.rms_norm_adaln(x, w, sc, sh, 1e-6, rows_per_cond=rpc, exact=True)
    t = np.repeat(sh.astype(np.float64), rpc, axis=0)[:rows]
    r = compare_fmt_bounded(host(out, fmt), ye, adaln_bound(hidden, ye, t))
    assert r["ok"], r


# ------------------------------------------------------------ residual add --

@pytest.mark.parametrize("fmt", ["f16", "f32"])
@pytest.mark.parametrize("rows,hidden", [(64, 3072), (33, 2048), (5, 24), (7, 13)])
def test_add_rms_norm(fmt, rows, hidden):
    seed = 7000 + rows + hidden
    x = synth.normal_bf16(seed, 0, rows * hidden, fmt=fmt).reshape(rows, hidden)
    r = synth.normal_bf16(seed, 5, rows * hidden, fmt=fmt).reshape(rows, hidden)
    w = synth.normal_bf16(seed, 2, hidden, 1.0, 0.1, fmt=fmt)
    whole, out = guarded(rows * hidden, fmt)
    hwhole, hout = guarded(rows * hidden, fmt)
    xd, rd, wd = dev(x), dev(r), dev(w)
    st = L.ltxk_add_rms_norm_dt(out.data_ptr(), hout.data_ptr(), xd.data_ptr(), rd.data_ptr(),
                                wd.data_ptr(), rows, hidden, 1e-6, FMTS[fmt][2], stream())
    assert st == L.OK, L.ltxk_status_string(st)
    torch.cuda.synchronize()
    check_guard(whole, rows * hidden, fmt)
    check_guard(hwhole, rows * hidden, fmt)
    y_ref, h_ref, ye = oracle.add_rms_norm(x, r, w, 1e-6, exact=True)
    ut = FMTS[fmt][3]
    assert np.array_equal(host(hout, fmt).view(ut), h_ref.reshape(-1).view(ut)), \
        "h must be bit-exact"
    if fmt == "f16":
        res = compare_fmt(host(out, fmt), y_ref.reshape(-1))
    else:
        res = compare_fmt_bounded(host(out, fmt), ye, (delta(hidden) + 4 * U) * np.abs(ye))
    assert res["ok"], res


# ----------------------------------------------------------------- helpers --

@pytest.mark.parametrize("fmt", ["f16", "f32"])
def test_torch_helpers(fmt):
    npt, tt = FMTS[fmt][0], FMTS[fmt][1]
    x = synth.normal_bf16(81, 0, 3 * 7 * 256, fmt=fmt).reshape(3, 7, 256)
    w = synth.normal_bf16(81, 2, 256, 1.0, 0.1, fmt=fmt)
    xt, wt = dev(x), dev(w)
    y = L.rms_norm(xt, wt)
    torch.cuda.synchronize()
    assert y.dtype == tt and y.shape == xt.shape
    check_plain(host(y, fmt), x.reshape(21, 256), w, 1e-6, fmt, "helper")
    y2, h = L.add_rms_norm(xt, xt, wt)
    torch.cuda.synchronize()
    assert y2.dtype == tt and h.dtype == tt
    with pytest.raises(TypeError):
        L.rms_norm(xt, wt.to(torch.bfloat16))
