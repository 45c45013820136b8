"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, on the
same seeded inputs, element by element.

Tolerance (from the definition of the output as one RNE rounding of the exact
value): at most 1 bf16 ulp between GPU and oracle on every element -- the
ordinal distance of oracle/compare.py.  The GPU computes in fp32 with a
relative error of a few 1e-6 (sum of squares, rsqrtf, Kahan-evaluated
rotation), far below the 2^-8 bf16 spacing, so a difference can only be a
neighbouring value near a rounding midpoint.

Covers every workload at full size (in the launch configuration the
benchmark times), small shapes that span several CTAs with ragged tails,
every kernel family (16-byte vector path, element-wise path), weight-less
calls, in-place calls, unaligned pointers, guard bands, non-default streams
and run-to-run determinism.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import rope_element_dit_gb300 as L
import synth
from oracle.compare import compare_bf16, compare_bf16_bounded

pytestmark = pytest.mark.gpu

THREADS = min(32, os.cpu_count() or 1)
CANARY = 0x7FC1          # a NaN pattern the kernels never write
GUARD = 64


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU parity tests need a CUDA device"
    torch.cuda.set_device(0)
    cap = torch.cuda.get_device_capability(0)
    assert cap == (10, 3), f"expected an sm_103 GPU, got {cap}"
    return torch.device("cuda:0")


@pytest.fixture(params=["registers", "tma"])
def path(request):
    """Run the test under each vectorised kernel family (the planner picks
    the TMA ring only where one warp can own a row; elsewhere both settings
    give the same kernel)."""
    value = {"registers": L.PATH_REGISTERS, "tma": L.PATH_TMA}[request.param]
    old = L.ltxk_set_path(value)
    yield request.param
    L.ltxk_set_path(old)


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def to_host(t):
    return t.cpu().numpy().view(np.uint16)


def guarded(n):
    """Device buffer of n bf16 with GUARD canary elements on each side;
    returns (whole, inner view).  The inner view starts 128 bytes in, so its
    16-byte alignment matches the allocation's."""
    whole = torch.full((n + 2 * GUARD,), CANARY, dtype=torch.int16, device="cuda")
    return whole, whole[GUARD:GUARD + n]


def check_guard(whole, n):
    h = to_host(whole)
    assert np.all(h[:GUARD] == CANARY) and np.all(h[GUARD + n:] == CANARY), \
        "kernel wrote outside its output"


def assert_parity(got, ref, what):
    r = compare_bf16(got, ref)
    assert r["ok"], f"{what}: {r}"
    return r


def compare_chunked(got, ref, what, chunk=1 << 26):
    got = got.reshape(-1)
    ref = ref.reshape(-1)
    total = {"elements": 0, "exact": 0, "one_ulp": 0}
    for s in range(0, got.size, chunk):
        r = assert_parity(got[s:s + chunk], ref[s:s + chunk], f"{what}[{s}:]")
        for k in total:
            total[k] += r[k]
    return total


def dptr(t):
    return None if t is None else t.data_ptr()


def stream_ptr():
    return torch.cuda.current_stream().cuda_stream


def gpu_rms_norm(x_dev, w_dev, rows, hidden, eps, out=None):
    if out is None:
        out = torch.empty(rows * hidden, dtype=torch.int16, device="cuda")
    st = L.ltxk_rms_norm(dptr(out), dptr(x_dev), dptr(w_dev), rows, hidden, eps,
                         stream_ptr())
    assert st == L.OK, L.ltxk_status_string(st)
    return out


def gpu_rope(x_dev, w_dev, c_dev, s_dev, rows, heads, D, mode, eps, seq_len=None,
             out=None):
    if out is None:
        out = torch.empty(rows * heads * D, dtype=torch.int16, device="cuda")
    if seq_len is None:
        st = L.ltxk_rms_norm_rope(dptr(out), dptr(x_dev), dptr(w_dev), dptr(c_dev),
                                  dptr(s_dev), rows, heads, D, mode, eps, stream_ptr())
    else:
        st = L.ltxk_rms_norm_rope_seq(dptr(out), dptr(x_dev), dptr(w_dev), dptr(c_dev),
                                      dptr(s_dev), rows, heads, D, mode, eps, seq_len,
                                      stream_ptr())
    assert st == L.OK, L.ltxk_status_string(st)
    return out


# ---------------------------------------------------------------- workloads --

ALL_CASES = [c for cases in synth.WORKLOADS.values() for c in cases
             if c.kind not in ("gelu", "geglu", "rope_pos")   # test_gpu_gelu.py, _rope_pos.py
             and c.dtype == "bf16"]                   # fp16 / fp32: test_gpu_dtypes.py


def adaln_bound(hidden, y_exact, shift_rows):
    """Bound on the GPU's fp32 error in n*(1+scale)+shift before rounding.

    n = (x*w)*inv_rms carries a relative error delta(H) from the fp32 sum of
    squares (at most H/64 + 40 chained additions), the mean, eps, rsqrtf
    (2 ulp) and the product; the shift can cancel n*(1+scale), so the bound
    is absolute: 2*delta*|n(1+s)| plus the roundings of 1+s and of the FMA."""
    delta = (hidden / 128 + 26) * 2.0 ** -24
    ns = np.abs(y_exact - shift_rows)
    return 2 * delta * ns + 2.0 ** -22 * (ns + np.abs(shift_rows))


def gpu_adaln(x_dev, w_dev, sc_dev, sh_dev, rows, hidden, rows_per_cond, eps, out=None):
    if out is None:
        out = torch.empty(rows * hidden, dtype=torch.int16, device="cuda")
    st = L.ltxk_rms_norm_adaln(dptr(out), dptr(x_dev), dptr(w_dev), dptr(sc_dev),
                               dptr(sh_dev), rows, hidden, rows_per_cond, eps, stream_ptr())
    assert st == L.OK, L.ltxk_status_string(st)
    return out


# At most this fraction of a full-size AdaLN workload's elements may need the
# bound's second clause (more than 1 ulp from the correctly rounded value):
# only where the shift nearly cancels n*(1+scale) does the fp32 error of n
# reach a bf16 spacing of the result.  Measured: 46 of 25.2 M.
ADALN_STRICT_CAP = 2.0 ** -16


def check_adaln(got_bits, x, w, scale, shift, rows_per_cond, eps, what, threads=1):
    """Bounded comparison with the oracle; returns the total counts."""
    rows, H = x.shape
    _, ye = oracle.rms_norm_adaln(x, w, scale, shift, eps, rows_per_cond=rows_per_cond,
                                  threads=threads, exact=True)
    t = np.repeat(oracle.widen_bf16(shift), rows_per_cond, axis=0)[:rows]
    got = got_bits.reshape(rows, H)
    step = max(1, (1 << 24) // H)
    tot = {"elements": 0, "exact": 0, "one_ulp": 0, "beyond_1ulp_within_bound": 0}
    for r0 in range(0, rows, step):
        r = compare_bf16_bounded(got[r0:r0 + step], ye[r0:r0 + step],
                                 adaln_bound(H, ye[r0:r0 + step], t[r0:r0 + step]))
        assert r["ok"], f"{what} rows {r0}+: {r}"
        for k in tot:
            tot[k] += r[k]
    return tot


@pytest.mark.parametrize("case", ALL_CASES, ids=[c.name for c in ALL_CASES])
def test_workload_full_size(case, path):
    inp = synth.make_inputs(case)
    x, w = inp["x"], inp["w"]
    n = case.rows * case.hidden
    whole, out = guarded(n)
    xd, wd = to_dev(x), (None if w is None else to_dev(w))
    if case.kind == "add_norm":
        hwhole, hout = guarded(n)
        rd = to_dev(inp["res"])
        st = L.ltxk_add_rms_norm(dptr(out), dptr(hout), dptr(xd), dptr(rd),
                                 dptr(wd), case.rows, case.hidden, case.eps, stream_ptr())
        assert st == L.OK
        torch.cuda.synchronize()
        check_guard(whole, n)
        check_guard(hwhole, n)
        y_ref, h_ref = oracle.add_rms_norm(x, inp["res"], w, case.eps, threads=THREADS)
        assert np.array_equal(to_host(hout), h_ref.ravel()), "h must be bit-exact"
        compare_chunked(to_host(out), y_ref, case.name)
        return
    if case.kind == "adaln":
        gpu_adaln(xd, wd, to_dev(inp["scale"]), to_dev(inp["shift"]), case.rows,
                  case.hidden, case.rows_per_cond, case.eps, out=out)
        torch.cuda.synchronize()
        check_guard(whole, n)
        r = check_adaln(to_host(out), x, w, inp["scale"], inp["shift"], case.rows_per_cond,
                        case.eps, case.name, threads=THREADS)
        assert r["beyond_1ulp_within_bound"] <= ADALN_STRICT_CAP * r["elements"], r
        assert L.ltxk_fault_status() == L.OK
        return
    if case.mode is None:
        gpu_rms_norm(xd, wd, case.rows, case.hidden, case.eps, out=out)
        ref = oracle.rms_norm(x, w, case.eps, threads=THREADS)
    else:
        cd = torch.from_numpy(inp["cos"]).cuda()
        sd = torch.from_numpy(inp["sin"]).cuda()
        mode = case.mode
        gpu_rope(xd, wd, cd, sd, case.rows, case.heads, case.head_dim, mode, case.eps,
                 seq_len=case.seq_len, out=out)
        ref = oracle.rms_norm_rope(x, w, inp["cos"], inp["sin"], case.heads,
                                   case.head_dim, mode, case.eps, threads=THREADS)
    torch.cuda.synchronize()
    check_guard(whole, n)
    stats = compare_chunked(to_host(out), ref, case.name)
    assert stats["elements"] == n
    if case.mode is not None:
        # the same result through per-row tables (the 11-argument call)
        reps = case.rows // case.seq_len
        cd = torch.from_numpy(np.concatenate([inp["cos"]] * reps)).cuda()
        sd = torch.from_numpy(np.concatenate([inp["sin"]] * reps)).cuda()
        out2 = gpu_rope(xd, wd, cd, sd, case.rows, case.heads, case.head_dim, case.mode,
                        case.eps)
        torch.cuda.synchronize()
        assert torch.equal(out2, out)
    assert L.ltxk_fault_status() == L.OK


# ---------------------------------------------------------- RMSNorm shapes --

NORM_SHAPES = [(1, 4), (3, 8), (37, 24), (9, 40), (1000, 264), (17, 2056),
               (1001, 3072), (33, 5120), (19, 8200), (3, 131072), (2, 131080),
               (2049, 2048), (5, 7), (4, 1), (9, 4096), (7, 6144), (5, 8192),
               (3, 12288), (3, 16384), (2, 24576), (2, 32768), (11, 2560)]


@pytest.mark.parametrize("rows,hidden", NORM_SHAPES)
@pytest.mark.parametrize("with_w", [True, False])
def test_rms_norm_shapes(rows, hidden, with_w, path):
    seed = 1000 + rows + hidden
    x = synth.normal_bf16(seed, 0, rows * hidden).reshape(rows, hidden)
    w = synth.normal_bf16(seed, 2, hidden, 1.0, 0.1) if with_w else None
    whole, out = guarded(rows * hidden)
    gpu_rms_norm(to_dev(x), None if w is None else to_dev(w), rows, hidden, 1e-6, out=out)
    torch.cuda.synchronize()
    check_guard(whole, rows * hidden)
    assert_parity(to_host(out), oracle.rms_norm(x, w, 1e-6), f"{rows}x{hidden}")


@pytest.mark.parametrize("rows,hidden", [(37, 3072), (5, 2056), (3, 24)])
def test_rms_norm_unaligned_pointers(rows, hidden):
    """Pointers 2 bytes off a 16-byte boundary take the element-wise kernel
    and give the same values."""
    x = synth.normal_bf16(7, 0, rows * hidden).reshape(rows, hidden)
    w = synth.normal_bf16(7, 2, hidden, 1.0, 0.1)
    xb = to_dev(np.concatenate([np.zeros(1, np.uint16), x.ravel()]))
    wb = to_dev(np.concatenate([np.zeros(1, np.uint16), w]))
    whole, out = guarded(rows * hidden + 1)
    gpu_rms_norm(xb[1:], wb[1:], rows, hidden, 1e-6, out=out[1:])
    torch.cuda.synchronize()
    check_guard(whole, rows * hidden + 1)
    assert_parity(to_host(out[1:]), oracle.rms_norm(x, w, 1e-6), "unaligned")


@pytest.mark.parametrize("rows,hidden", [(99, 3072), (7, 5120), (5, 24), (3, 131080)])
def test_rms_norm_in_place(rows, hidden, path):
    x = synth.uniform_bf16(8, 0, rows * hidden, -4, 4).reshape(rows, hidden)
    w = synth.normal_bf16(8, 2, hidden, 1.0, 0.1)
    xd = to_dev(x)
    gpu_rms_norm(xd, to_dev(w), rows, hidden, 1e-5, out=xd)
    torch.cuda.synchronize()
    assert_parity(to_host(xd), oracle.rms_norm(x, w, 1e-5), "in place")


def test_rms_norm_eps_and_scale_extremes():
    rows, hidden = 64, 2048
    x = synth.normal_bf16(9, 0, rows * hidden).reshape(rows, hidden)
    # row r scaled by 2^(r-32), i.e. 2^-32 .. 2^31: stresses eps against the
    # mean square while every square stays inside the fp32 range (the
    # kernel's sum of squares is fp32 by definition)
    k = np.arange(rows) - rows // 2
    xs = (x.astype(np.int32) + (k[:, None] << 7)).astype(np.uint16)
    for eps in (0.0, 1e-6, 1.0):
        out = gpu_rms_norm(to_dev(xs), None, rows, hidden, eps)
        torch.cuda.synchronize()
        assert_parity(to_host(out), oracle.rms_norm(xs, None, eps), f"eps={eps}")


def test_rms_norm_zero_rows_and_zero_input():
    x = np.zeros((8, 2048), np.uint16)
    out = gpu_rms_norm(to_dev(x), None, 8, 2048, 1e-6)
    torch.cuda.synchronize()
    assert np.all(to_host(out) == 0)
    assert L.ltxk_rms_norm(out.data_ptr(), out.data_ptr(), None, 0, 2048, 1e-6,
                           stream_ptr()) == L.OK


def test_rms_norm_side_stream_and_determinism(path):
    rows, hidden = 4096, 3072
    x = synth.normal_bf16(10, 0, rows * hidden).reshape(rows, hidden)
    w = synth.normal_bf16(10, 2, hidden, 1.0, 0.1)
    xd, wd = to_dev(x), to_dev(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = gpu_rms_norm(xd, wd, rows, hidden, 1e-6)
        b = gpu_rms_norm(xd, wd, rows, hidden, 1e-6)
    s.synchronize()
    assert torch.equal(a, b)
    assert_parity(to_host(a), oracle.rms_norm(x, w, 1e-6, threads=THREADS), "stream")


# ------------------------------------------------------------- fused shapes --

ROPE_SHAPES = [  # (rows, heads, head_dim, seq_len)
    (5, 1, 2, 5), (6, 1, 4, 3), (10, 2, 8, 4), (33, 3, 16, 11), (70, 4, 64, 24),
    (16, 32, 128, 8), (9, 2, 6, 9), (21, 5, 48, 7), (13, 2, 40, 13),
    (4, 64, 256, 2), (3, 80, 128, 1),
    (5003, 8, 64, 61),   # several rows per warp of the persistent (pipelined) grid
]


@pytest.mark.parametrize("rows,heads,D,seq_len", ROPE_SHAPES)
@pytest.mark.parametrize("mode", [0, 1])
def test_rope_shapes(rows, heads, D, seq_len, mode, path):
    H = heads * D
    seed = 2000 + rows + H + mode
    x = synth.normal_bf16(seed, 0, rows * H).reshape(rows, H)
    w = synth.normal_bf16(seed, 2, H, 1.0, 0.1)
    cos, sin = synth.rope_table_1d(seq_len, D)
    whole, out = guarded(rows * H)
    gpu_rope(to_dev(x), to_dev(w), torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda(),
             rows, heads, D, mode, 1e-6, seq_len=seq_len, out=out)
    torch.cuda.synchronize()
    check_guard(whole, rows * H)
    ref = oracle.rms_norm_rope(x, w, cos, sin, heads, D, mode, 1e-6)
    assert_parity(to_host(out), ref, f"rope {rows}x{heads}x{D} mode {mode}")


@pytest.mark.parametrize("mode", [0, 1])
def test_rope_unaligned_tables_and_no_weight(mode):
    rows, heads, D, S = 40, 4, 64, 10
    H = heads * D
    x = synth.normal_bf16(11, 0, rows * H).reshape(rows, H)
    cos, sin = synth.rope_table_1d(S, D)
    # tables 4 bytes past a 16-byte boundary: element-wise kernel
    cb = torch.from_numpy(np.concatenate([np.zeros(1, np.float32), cos.ravel()])).cuda()
    sb = torch.from_numpy(np.concatenate([np.zeros(1, np.float32), sin.ravel()])).cuda()
    out = gpu_rope(to_dev(x), None, cb[1:], sb[1:], rows, heads, D, mode, 1e-6, seq_len=S)
    torch.cuda.synchronize()
    ref = oracle.rms_norm_rope(x, None, cos, sin, heads, D, mode, 1e-6)
    assert_parity(to_host(out), ref, "unaligned tables")


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("heads,D", [(32, 128), (2, 6)])
def test_rope_in_place(mode, heads, D, path):
    rows, S = 48, 16
    H = heads * D
    x = synth.normal_bf16(12, 0, rows * H).reshape(rows, H)
    w = synth.normal_bf16(12, 2, H, 1.0, 0.1)
    cos, sin = synth.rope_table_1d(S, D)
    xd = to_dev(x)
    gpu_rope(xd, to_dev(w), torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda(),
             rows, heads, D, mode, 1e-6, seq_len=S, out=xd)
    torch.cuda.synchronize()
    ref = oracle.rms_norm_rope(x, w, cos, sin, heads, D, mode, 1e-6)
    assert_parity(to_host(xd), ref, "rope in place")


@pytest.mark.parametrize("mode", [0, 1])
def test_rope_position_zero_equals_plain_norm(mode, path):
    """cos = 1, sin = 0 at position 0: the fused output of those rows is the
    plain RMSNorm output (bit for bit where both kernels sum the squares in
    the same order)."""
    c = synth.ROPE_INTERLEAVED[0] if mode == 0 else synth.ROPE_SPLIT[0]
    rows = 2 * c.seq_len if mode == 0 else c.seq_len
    x = synth.make_x(c)
    w = synth.make_w(c)
    cos, sin = synth.make_tables(c)
    xd, wd = to_dev(x), to_dev(w)
    fused = gpu_rope(xd, wd, torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda(),
                     rows, c.heads, c.head_dim, mode, c.eps, seq_len=c.seq_len)
    plain = gpu_rms_norm(xd, wd, rows, c.hidden, c.eps)
    torch.cuda.synchronize()
    f = to_host(fused).reshape(rows, c.hidden)
    p = to_host(plain).reshape(rows, c.hidden)
    for r in range(0, rows, c.seq_len):
        if mode == 0:
            # same slot map as the plain kernel: identical sums, identical bits
            assert np.array_equal(f[r], p[r])
        else:
            # split-half pairs slots differently, so the fp32 sum of squares
            # may round differently in its last bit
            assert_parity(f[r], p[r], "position 0, split-half")


def test_rope_cancellation_stress(path):
    """Tables chosen so that a*c and b*s nearly cancel: the rotation is
    evaluated with a compensated difference, so even outputs far smaller
    than their inputs stay within 1 ulp."""
    rows, heads, D = 64, 8, 64
    H = heads * D
    P = D // 2
    x = synth.normal_bf16(13, 0, rows * H).reshape(rows, H)
    xv = synth.bf16_bits_to_f32(x).astype(np.float64).reshape(rows, heads, D)
    # per row r, choose the angle that zeroes pair 0 of head 0 exactly in
    # real arithmetic (tan = a/b); fp32 rounding of the table leaves a tiny
    # residue that the GPU must get right.
    for mode in (0, 1):
        if mode == 0:
            a, b = xv[:, 0, 0], xv[:, 0, 1]
        else:
            a, b = xv[:, 0, 0], xv[:, 0, P]
        theta = np.arctan2(a, b)     # a cos - b sin = 0
        ang = theta[:, None] + np.zeros((rows, P))
        cos = np.cos(ang).astype(np.float32)
        sin = np.sin(ang).astype(np.float32)
        out = gpu_rope(to_dev(x), None, torch.from_numpy(cos).cuda(),
                       torch.from_numpy(sin).cuda(), rows, heads, D, mode, 1e-6)
        torch.cuda.synchronize()
        ref = oracle.rms_norm_rope(x, None, cos, sin, heads, D, mode, 1e-6)
        assert_parity(to_host(out), ref, f"cancellation mode {mode}")


def test_binding_helpers_match_abi():
    rows, H = 300, 4096
    x = synth.normal_bf16(14, 0, rows * H).reshape(rows, H)
    w = synth.normal_bf16(14, 2, H, 1.0, 0.1)
    xt = to_dev(x).view(torch.bfloat16)
    wt = to_dev(w).view(torch.bfloat16)
    y = L.rms_norm(xt, wt, 1e-6)
    cos, sin = synth.rope_table_1d(rows, 128)
    yr = L.rms_norm_rope(xt, wt, torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda(),
                         32, 128, L.ROPE_INTERLEAVED, 1e-6)
    torch.cuda.synchronize()
    assert_parity(y.view(torch.int16).cpu().numpy().view(np.uint16),
                  oracle.rms_norm(x, w, 1e-6), "helper")
    assert_parity(yr.view(torch.int16).cpu().numpy().view(np.uint16),
                  oracle.rms_norm_rope(x, w, cos, sin, 32, 128, 0, 1e-6), "helper rope")
    with pytest.raises(L.LtxkError):
        L.rms_norm_rope(xt, wt, torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda(),
                        32, 128, 7, 1e-6)


# ------------------------------------------------------------ bounded waits --

def test_tma_wait_runs_out_and_context_survives():
    """The TMA-ring kernel's waits are bounded: with the bulk copy of each
    warp's first row never issued, every such wait gives up after the limit,
    the fault word is set, and the device stays usable."""
    rows, hidden = 4 * 152 * 2 * 8, 1024      # several rows per warp
    x = synth.normal_bf16(15, 0, rows * hidden).reshape(rows, hidden)
    xd = to_dev(x)
    out = torch.zeros(rows * hidden, dtype=torch.int16, device="cuda")
    assert L.ltxk_fault_status() == L.OK
    st = L.ltxk_diag_missing_copy(out.data_ptr(), xd.data_ptr(), rows, hidden,
                                  50_000_000, stream_ptr())
    assert st == L.OK
    assert L.ltxk_fault_status() == L.ERR_TIMEOUT
    assert L.ltxk_fault_status() == L.OK          # cleared by the read
    # the context still works and the normal path is still exact
    y = gpu_rms_norm(xd, None, rows, hidden, 1e-6)
    torch.cuda.synchronize()
    assert_parity(to_host(y), oracle.rms_norm(x, None, 1e-6), "after timeout")
    assert L.ltxk_fault_status() == L.OK


# ------------------------------------------------------------------ AdaLN --

ADALN_SHAPES = [  # (rows, hidden, rows_per_cond, with_w)
    (6, 4, 3, False), (7, 24, 3, True), (33, 264, 11, False), (100, 2048, 25, True),
    (1001, 3072, 1000, False), (64, 5120, 64, True), (9, 4096, 1, False),
    (5, 7, 2, True), (3, 131080, 2, False), (37, 2056, 10, True)]


@pytest.mark.parametrize("rows,hidden,rpc,with_w", ADALN_SHAPES)
def test_adaln_shapes(rows, hidden, rpc, with_w):
    seed = 3000 + rows + hidden
    n_cond = -(-rows // rpc)
    x = synth.normal_bf16(seed, 0, rows * hidden).reshape(rows, hidden)
    w = synth.normal_bf16(seed, 2, hidden, 1.0, 0.1) if with_w else None
    sc = synth.normal_bf16(seed, 3, n_cond * hidden, 0.0, 0.5).reshape(n_cond, hidden)
    sh = synth.normal_bf16(seed, 4, n_cond * hidden, 0.0, 0.5).reshape(n_cond, hidden)
    whole, out = guarded(rows * hidden)
    gpu_adaln(to_dev(x), None if w is None else to_dev(w), to_dev(sc), to_dev(sh), rows,
              hidden, rpc, 1e-6, out=out)
    torch.cuda.synchronize()
    check_guard(whole, rows * hidden)
    check_adaln(to_host(out), x, w, sc, sh, rpc, 1e-6, f"adaln {rows}x{hidden}/{rpc}")


def test_adaln_unaligned_and_in_place():
    rows, hidden, rpc = 40, 3072, 20
    x = synth.normal_bf16(51, 0, rows * hidden).reshape(rows, hidden)
    sc = synth.normal_bf16(51, 3, 2 * hidden, 0.0, 0.5).reshape(2, hidden)
    sh = synth.normal_bf16(51, 4, 2 * hidden, 0.0, 0.5).reshape(2, hidden)
    # scale 2 bytes off a 16-byte boundary: element-wise kernel
    scb = to_dev(np.concatenate([np.zeros(1, np.uint16), sc.ravel()]))
    out = gpu_adaln(to_dev(x), None, scb[1:], to_dev(sh), rows, hidden, rpc, 1e-6)
    torch.cuda.synchronize()
    check_adaln(to_host(out), x, None, sc, sh, rpc, 1e-6, "adaln unaligned")
    xd = to_dev(x)
    gpu_adaln(xd, None, to_dev(sc), to_dev(sh), rows, hidden, rpc, 1e-6, out=xd)
    torch.cuda.synchronize()
    check_adaln(to_host(xd), x, None, sc, sh, rpc, 1e-6, "adaln in place")


def test_adaln_zero_modulation_equals_rms_norm():
    rows, hidden = 257, 3072
    x = synth.normal_bf16(52, 0, rows * hidden).reshape(rows, hidden)
    w = synth.normal_bf16(52, 2, hidden, 1.0, 0.1)
    zero = torch.zeros(hidden, dtype=torch.int16, device="cuda")
    xd, wd = to_dev(x), to_dev(w)
    a = gpu_adaln(xd, wd, zero, zero, rows, hidden, rows, 1e-6)
    b = gpu_rms_norm(xd, wd, rows, hidden, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_adaln_binding_helper():
    B, S, H = 2, 48, 2048
    x = synth.normal_bf16(53, 0, B * S * H).reshape(B * S, H)
    sc = synth.normal_bf16(53, 3, B * H, 0.0, 0.5).reshape(B, H)
    sh = synth.normal_bf16(53, 4, B * H, 0.0, 0.5).reshape(B, H)
    y = L.rms_norm_adaln(to_dev(x).view(torch.bfloat16).reshape(B, S, H), None,
                         to_dev(sc).view(torch.bfloat16), to_dev(sh).view(torch.bfloat16))
    torch.cuda.synchronize()
    check_adaln(y.view(torch.int16).cpu().numpy().view(np.uint16).reshape(B * S, H), x,
                None, sc, sh, S, 1e-6, "adaln helper")


# --------------------------------------------------------- host pipeline --

# pinned: page-locked host buffers take the zero-copy kernel; pageable ones
# (and pinned ones under the TMA path setting) the staged pipeline
@pytest.mark.parametrize("rows,hidden,slot_rows,n_streams,pinned", [
    (4099, 3072, 512, 3, True), (1000, 2048, 1, 2, True), (37, 264, 5, 3, False),
    (16384, 3072, 4096, 3, True), (9, 24, 100, 1, True), (4099, 3072, 512, 3, False),
    (1000, 2048, 1, 2, False), (2049, 2056, 300, 2, "staged")])
def test_host_pipeline_matches_device_call(rows, hidden, slot_rows, n_streams, pinned):
    x = synth.normal_bf16(61, 0, rows * hidden).reshape(rows, hidden)
    w = synth.normal_bf16(61, 2, hidden, 1.0, 0.1)
    xh = torch.from_numpy(x.view(np.int16).copy())
    yh = torch.full_like(xh, 0x7FC1)
    old = None
    if pinned:
        xh, yh = xh.pin_memory(), yh.pin_memory()
    if pinned == "staged":
        old = L.ltxk_set_path(L.PATH_TMA)
    wd = to_dev(w)
    slot = (slot_rows * hidden * 2 + 255) // 256 * 256
    staging = torch.empty(n_streams * slot, dtype=torch.uint8, device="cuda")
    streams = [torch.cuda.Stream() for _ in range(n_streams)]
    st = L.ltxk_rms_norm_host(yh.data_ptr(), xh.data_ptr(), wd.data_ptr(), rows, hidden,
                              1e-6, staging.data_ptr(), staging.numel(),
                              [s.cuda_stream for s in streams], n_streams)
    for s in streams:
        s.synchronize()
    if old is not None:
        L.ltxk_set_path(old)
    assert st == L.OK
    ref = gpu_rms_norm(to_dev(x), wd, rows, hidden, 1e-6)
    torch.cuda.synchronize()
    assert np.array_equal(yh.numpy().view(np.uint16).ravel(), to_host(ref))


@pytest.mark.parametrize("pinned", [True, False])
def test_host_pipeline_in_place(pinned):
    """out_host == x_host on both the zero-copy and the staged branch."""
    rows, hidden = 777, 3072
    x = synth.normal_bf16(62, 0, rows * hidden).reshape(rows, hidden)
    xh = torch.from_numpy(x.view(np.int16).copy())
    if pinned:
        xh = xh.pin_memory()
    staging = torch.empty(2 * (4 << 20), dtype=torch.uint8, device="cuda")
    streams = [torch.cuda.Stream() for _ in range(2)]
    st = L.ltxk_rms_norm_host(xh.data_ptr(), xh.data_ptr(), None, rows, hidden, 1e-6,
                              staging.data_ptr(), staging.numel(),
                              [s.cuda_stream for s in streams], 2)
    for s in streams:
        s.synchronize()
    assert st == L.OK
    assert_parity(xh.numpy().view(np.uint16).ravel(), oracle.rms_norm(x, None, 1e-6), "in place")


def test_host_pipeline_helper():
    rows, hidden = 3000, 2048
    x = synth.normal_bf16(62, 0, rows * hidden).reshape(rows, hidden)
    xh = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    y = L.rms_norm_host(xh, None, 1e-6)
    assert_parity(y.view(torch.int16).numpy().view(np.uint16), oracle.rms_norm(x, None, 1e-6),
                  "host helper")


# ------------------------------------------------------------ residual add --

ADD_SHAPES = [(1, 4), (3, 24), (37, 264), (1000, 2048), (1001, 3072), (33, 5120),
              (9, 4096), (5, 7), (2, 131080), (4, 8192)]


@pytest.mark.parametrize("rows,hidden", ADD_SHAPES)
@pytest.mark.parametrize("with_w", [True, False])
def test_add_rms_norm_shapes(rows, hidden, with_w):
    seed = 5000 + rows + hidden
    x = synth.normal_bf16(seed, 0, rows * hidden).reshape(rows, hidden)
    r = synth.normal_bf16(seed, 5, rows * hidden).reshape(rows, hidden)
    w = synth.normal_bf16(seed, 2, hidden, 1.0, 0.1) if with_w else None
    yw, y = guarded(rows * hidden)
    hw, h = guarded(rows * hidden)
    # keep every input tensor referenced until the kernel has run: a freed
    # temporary's block would be handed to the next allocation
    xd, rd = to_dev(x), to_dev(r)
    wd = None if w is None else to_dev(w)
    st = L.ltxk_add_rms_norm(y.data_ptr(), h.data_ptr(), xd.data_ptr(), rd.data_ptr(),
                             dptr(wd), rows, hidden, 1e-6, stream_ptr())
    assert st == L.OK
    torch.cuda.synchronize()
    check_guard(yw, rows * hidden)
    check_guard(hw, rows * hidden)
    y_ref, h_ref = oracle.add_rms_norm(x, r, w, 1e-6)
    assert np.array_equal(to_host(h), h_ref.ravel())
    assert_parity(to_host(y), y_ref, f"add norm {rows}x{hidden}")


def test_add_rms_norm_in_place_residual_stream():
    """residual_out == residual (update the stream) and out == x."""
    rows, hidden = 515, 3072
    x = synth.normal_bf16(71, 0, rows * hidden).reshape(rows, hidden)
    r = synth.normal_bf16(71, 5, rows * hidden).reshape(rows, hidden)
    xd, rd = to_dev(x), to_dev(r)
    st = L.ltxk_add_rms_norm(xd.data_ptr(), rd.data_ptr(), xd.data_ptr(), rd.data_ptr(), None,
                             rows, hidden, 1e-6, stream_ptr())
    assert st == L.OK
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.add_rms_norm(x, r, None, 1e-6)
    assert np.array_equal(to_host(rd).ravel(), h_ref.ravel())
    assert_parity(to_host(xd), y_ref, "add norm in place")


def test_add_rms_norm_unaligned_and_helper():
    rows, hidden = 40, 2048
    x = synth.normal_bf16(72, 0, rows * hidden).reshape(rows, hidden)
    r = synth.normal_bf16(72, 5, rows * hidden).reshape(rows, hidden)
    rb = to_dev(np.concatenate([np.zeros(1, np.uint16), r.ravel()]))
    y = torch.empty(rows * hidden, dtype=torch.int16, device="cuda")
    h = torch.empty_like(y)
    xd = to_dev(x)
    st = L.ltxk_add_rms_norm(y.data_ptr(), h.data_ptr(), xd.data_ptr(),
                             rb[1:].data_ptr(), None, rows, hidden, 1e-6, stream_ptr())
    assert st == L.OK
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.add_rms_norm(x, r, None, 1e-6)
    assert np.array_equal(to_host(h), h_ref.ravel())
    assert_parity(to_host(y), y_ref, "add norm unaligned")
    yt, ht = L.add_rms_norm(to_dev(x).view(torch.bfloat16), to_dev(r).view(torch.bfloat16))
    torch.cuda.synchronize()
    assert np.array_equal(ht.view(torch.int16).cpu().numpy().view(np.uint16).ravel(),
                          h_ref.ravel())
    assert_parity(yt.view(torch.int16).cpu().numpy().view(np.uint16), y_ref, "add norm helper")
