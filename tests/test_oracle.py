"""Pins for the fp64 CPU oracle, checked against what the definition and the
mathematics fix -- never against the CUDA path.

Each test is chosen so that a plausible slip in the oracle fails it:
  * rounding: brute force over every bfloat16 pattern, midpoints, ties,
    overflow and subnormals; plus PyTorch's binary32 -> bfloat16 conversion
    (a library routine) on binary32 inputs;
  * RMSNorm: hand cases at hidden = 4 (tests/golden), the unit-RMS closed
    form (mean over exactly H), exact power-of-two scale invariance (eps
    inside the root, scaled by 1/alpha^2), a first-order expansion in eps,
    and PyTorch's float64 library RMSNorm;
  * RoPE: hand cases (pair indices, signs, table row per position), the
    identity at angle 0, quarter and half turns, pair-norm preservation and
    the permutation that maps split-half pairing onto interleaved pairing.
"""
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases_h4.txt")


def f32_to_bits(v):
    return (np.asarray(v, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bits_of(values):
    """bf16 bit patterns of values that are exactly representable."""
    f = np.asarray(values, np.float32)
    assert np.all((f.view(np.uint32) & 0xFFFF) == 0)
    return f32_to_bits(f)


# ---------------------------------------------------------------- rounding --

def test_widen_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle_mod.widen_bf16(bits)
    with np.errstate(invalid="ignore"):
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(vals), nan)
    assert np.array_equal(vals[~nan], ref[~nan])


def test_round_identity_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle_mod.widen_bf16(bits)
    back = oracle_mod.round_bf16(vals)
    finite = ~np.isnan(vals)
    assert np.array_equal(back[finite], bits[finite])
    # NaN stays NaN (quiet, sign kept)
    nb = back[~finite]
    assert np.all((nb & 0x7F80) == 0x7F80) and np.all((nb & 0x7F) != 0)


def test_round_midpoints_ties_to_even(oracle_mod):
    # consecutive positive finite patterns b, b+1 (b+1 may be +inf = 0x7F80)
    b = np.arange(0, 0x7F80, dtype=np.uint16)
    lo = oracle_mod.widen_bf16(b)
    hi = oracle_mod.widen_bf16((b + 1).astype(np.uint16))
    hi[-1] = 2.0 ** 128                     # the value "after" the max finite
    mid = (lo + hi) / 2                     # exact in binary64
    even = np.where(b % 2 == 0, b, b + 1).astype(np.uint16)
    assert np.array_equal(oracle_mod.round_bf16(mid), even)
    delta = (hi - lo) * 2.0 ** -20
    assert np.array_equal(oracle_mod.round_bf16(mid + delta), (b + 1).astype(np.uint16))
    assert np.array_equal(oracle_mod.round_bf16(mid - delta), b)
    # negative side mirrors the positive side
    assert np.array_equal(oracle_mod.round_bf16(-mid), even | np.uint16(0x8000))


def test_round_special_values(oracle_mod):
    r = oracle_mod.round_bf16
    cases = [
        (0.0, 0x0000), (-0.0, 0x8000), (np.inf, 0x7F80), (-np.inf, 0xFF80),
        (2.0 ** -133, 0x0001),             # smallest subnormal
        (2.0 ** -134, 0x0000),             # half of it: tie -> even (0)
        (1.5 * 2.0 ** -134, 0x0001),
        (3.0 * 2.0 ** -134, 0x0002),       # tie between 1 and 2 -> 2
        (2.0 ** -126, 0x0080),             # smallest normal
        ((2 - 2 ** -7) * 2.0 ** 127, 0x7F7F),   # largest finite
        ((2 - 2 ** -8) * 2.0 ** 127, 0x7F80),   # its upper midpoint -> inf
        (1e300, 0x7F80),
        (1.0 + 2 ** -8, 0x3F80),           # tie, 1.0 is even
        (1.0 + 3 * 2 ** -8, 0x3F82),       # tie, 1+2^-6 (..010) is even
        (1.0 + 2 ** -8 + 2 ** -50, 0x3F81),  # just above the tie
    ]
    vals = np.array([v for v, _ in cases], np.float64)
    got = r(vals)
    assert [int(g) for g in got] == [b for _, b in cases]


def test_round_direct_not_through_binary32(oracle_mod):
    # A binary64 just above a bf16 midpoint whose nearest binary32 IS the
    # midpoint: direct rounding goes up, rounding through binary32 would tie
    # to even (down).
    v = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert np.float64(np.float32(v)) == 1.0 + 2.0 ** -8
    assert int(oracle_mod.round_bf16(np.array([v]))[0]) == 0x3F81


def test_round_matches_torch_on_binary32(oracle_mod):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    f = (rng.standard_normal(1 << 18)
         * np.exp2(rng.integers(-140, 128, 1 << 18))).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.round_bf16(f.astype(np.float64))
    ok = np.isfinite(f)
    assert np.array_equal(got[ok], ref[ok])


# ------------------------------------------------------------- hand cases --

def _parse_golden():
    cases = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = [s.strip() for s in line.split(" | ")]
        name, kind, eps, xs, ws, tab, hd, exact, bits = f
        rows = [list(map(float, r.split())) for r in xs.split(";")]
        x = np.array(rows, np.float64)
        w = None if ws == "-" else np.array(list(map(float, ws.split())))
        cos = sin = None
        if tab != "-":
            c, s = tab.split(";")
            cos = np.array(list(map(float, c.split())), np.float32)
            sin = np.array(list(map(float, s.split())), np.float32)
        heads = head_dim = None
        if hd != "-":
            heads, head_dim = map(int, hd.split(","))
        cases.append(dict(
            name=name, kind=kind, eps=float(eps), x=x, w=w, cos=cos, sin=sin,
            heads=heads, head_dim=head_dim,
            exact=np.array(list(map(float, exact.split()))).reshape(x.shape),
            bits=np.array([int(b, 16) for b in bits.split()],
                          np.uint16).reshape(x.shape)))
    return cases


@pytest.mark.parametrize("case", _parse_golden(), ids=lambda c: c["name"])
def test_hand_cases(oracle_mod, case):
    x = bits_of(case["x"])
    w = None if case["w"] is None else bits_of(case["w"])
    if case["kind"] == "norm":
        y, ye = oracle_mod.rms_norm(x, w, case["eps"], exact=True)
    else:
        mode = (oracle_mod.INTERLEAVED if case["kind"] == "rope_interleaved"
                else oracle_mod.SPLIT_HALF)
        y, ye = oracle_mod.rms_norm_rope(
            x, w, case["cos"], case["sin"], case["heads"], case["head_dim"],
            mode, case["eps"], exact=True)
    assert np.array_equal(y, case["bits"]), [hex(v) for v in y.ravel()]
    np.testing.assert_allclose(ye, case["exact"], rtol=4e-16, atol=1e-300)


def test_eps_first_order(oracle_mod):
    # x = (3, 4, 0, 0): y0 = 1.2 (1 + e/6.25)^(-1/2) = 1.2 - 0.096 e + O(e^2).
    # eps outside the root would give 1.2 - 0.48 e instead.
    e = float(np.float32(1e-6))
    x = bits_of([[3, 4, 0, 0]])
    _, ye = oracle_mod.rms_norm(x, None, 1e-6, exact=True)
    assert abs(ye[0, 0] - (1.2 - 0.096 * e)) < 2e-14
    assert abs(ye[0, 1] - (1.6 - 0.128 * e)) < 2e-14


# --------------------------------------------------------- RMSNorm pins --

def _rows(seed, rows, H, dist="normal"):
    if dist == "normal":
        return synth.normal_bf16(seed, 0, rows * H).reshape(rows, H)
    return synth.uniform_bf16(seed, 0, rows * H, -4, 4).reshape(rows, H)


@pytest.mark.parametrize("H", [4, 24, 2048, 5120])
def test_unit_rms_closed_form(oracle_mod, H):
    x = _rows(11, 16, H)
    _, ye = oracle_mod.rms_norm(x, None, 0.0, exact=True)
    np.testing.assert_allclose((ye ** 2).mean(axis=1), 1.0, rtol=1e-13)
    # with eps: mean(n^2) = ms / (ms + eps)
    eps = 0.25
    _, ye = oracle_mod.rms_norm(x, None, eps, exact=True)
    ms = (oracle_mod.widen_bf16(x) ** 2).mean(axis=1)
    np.testing.assert_allclose((ye ** 2).mean(axis=1), ms / (ms + eps), rtol=1e-13)


@pytest.mark.parametrize("k", [-3, 1, 5])
def test_scale_invariance_exact(oracle_mod, k):
    x = _rows(12, 8, 264)
    w = synth.normal_bf16(12, 2, 264, 1.0, 0.1)
    xs = (x.astype(np.int32) + (k << 7)).astype(np.uint16)   # x * 2^k, exact
    assert np.array_equal(oracle_mod.widen_bf16(xs), oracle_mod.widen_bf16(x) * 2.0 ** k)
    # eps = 0: identical output
    y0, e0 = oracle_mod.rms_norm(x, w, 0.0, exact=True)
    y1, e1 = oracle_mod.rms_norm(xs, w, 0.0, exact=True)
    assert np.array_equal(y0, y1) and np.array_equal(e0, e1)
    # eps > 0: n(2^k x; eps) == n(x; eps / 4^k) exactly
    eps = float(np.float32(1e-3))
    _, ea = oracle_mod.rms_norm(xs, w, eps, exact=True)
    _, eb = oracle_mod.rms_norm(x, w, eps / 4.0 ** k, exact=True)
    assert np.array_equal(ea, eb)


def test_weight_none_is_ones(oracle_mod):
    x = _rows(13, 4, 40)
    ones = bits_of(np.ones(40))
    assert np.array_equal(oracle_mod.rms_norm(x, None, 1e-6),
                          oracle_mod.rms_norm(x, ones, 1e-6))


def test_matches_torch_rms_norm_fp64(oracle_mod):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    if not hasattr(F, "rms_norm"):
        pytest.skip("torch without rms_norm")
    for H, eps in [(24, 1e-6), (2048, 1e-5), (3072, 1e-6)]:
        x = _rows(14, 8, H, "uniform")
        w = synth.normal_bf16(14, 2, H, 1.0, 0.1)
        _, ye = oracle_mod.rms_norm(x, w, eps, exact=True)
        xt = torch.from_numpy(oracle_mod.widen_bf16(x))
        wt = torch.from_numpy(oracle_mod.widen_bf16(w))
        ref = F.rms_norm(xt, (H,), wt, eps=float(np.float32(eps))).numpy()
        np.testing.assert_allclose(ye, ref, rtol=1e-12, atol=1e-300)


def test_threaded_rows_identical(oracle_mod):
    x = _rows(15, 37, 96)
    w = synth.normal_bf16(15, 2, 96, 1.0, 0.1)
    assert np.array_equal(oracle_mod.rms_norm(x, w, 1e-6, threads=1),
                          oracle_mod.rms_norm(x, w, 1e-6, threads=5))
    c, s = synth.rope_table_1d(7, 8)
    a = oracle_mod.rms_norm_rope(x, w, c, s, 12, 8, 0, 1e-6, threads=1)
    b = oracle_mod.rms_norm_rope(x, w, c, s, 12, 8, 0, 1e-6, threads=4)
    assert np.array_equal(a, b)


# ------------------------------------------------------------- RoPE pins --

def _const_tables(rows, P, c, s):
    return (np.full((rows, P), c, np.float32), np.full((rows, P), s, np.float32))


@pytest.mark.parametrize("mode", [0, 1])
def test_rope_identity_at_angle_zero(oracle_mod, mode):
    heads, D = 4, 16
    x = _rows(21, 9, heads * D)
    w = synth.normal_bf16(21, 2, heads * D, 1.0, 0.1)
    c, s = _const_tables(3, D // 2, 1.0, 0.0)
    y, ye = oracle_mod.rms_norm_rope(x, w, c, s, heads, D, mode, 1e-6, exact=True)
    yn, yne = oracle_mod.rms_norm(x, w, 1e-6, exact=True)
    assert np.array_equal(y, yn) and np.array_equal(ye, yne)


@pytest.mark.parametrize("mode", [0, 1])
def test_rope_quarter_and_half_turn(oracle_mod, mode):
    heads, D = 3, 8
    P = D // 2
    x = _rows(22, 5, heads * D)
    _, n = oracle_mod.rms_norm(x, None, 1e-6, exact=True)
    n = n.reshape(5, heads, D)
    if mode == 0:
        a, b = n[..., 0::2], n[..., 1::2]
    else:
        a, b = n[..., :P], n[..., P:]
    # quarter turn (c = 0, s = 1): (a, b) -> (-b, a)
    c, s = _const_tables(1, P, 0.0, 1.0)
    _, q = oracle_mod.rms_norm_rope(x, None, c, s, heads, D, mode, 1e-6, exact=True)
    q = q.reshape(5, heads, D)
    qa, qb = (q[..., 0::2], q[..., 1::2]) if mode == 0 else (q[..., :P], q[..., P:])
    assert np.array_equal(qa, -b) and np.array_equal(qb, a)
    # half turn (c = -1, s = 0): negation
    c, s = _const_tables(1, P, -1.0, 0.0)
    _, hh = oracle_mod.rms_norm_rope(x, None, c, s, heads, D, mode, 1e-6, exact=True)
    assert np.array_equal(hh.reshape(5, heads, D), -n)


@pytest.mark.parametrize("mode", [0, 1])
def test_rope_preserves_pair_norm(oracle_mod, mode):
    heads, D = 4, 32
    P = D // 2
    x = _rows(23, 64, heads * D)
    w = synth.normal_bf16(23, 2, heads * D, 1.0, 0.1)
    cos, sin = synth.rope_table_1d(64, D)
    _, n = oracle_mod.rms_norm(x, w, 1e-6, exact=True)
    _, r = oracle_mod.rms_norm_rope(x, w, cos, sin, heads, D, mode, 1e-6, exact=True)
    n = n.reshape(64, heads, D)
    r = r.reshape(64, heads, D)
    if mode == 0:
        n2 = n[..., 0::2] ** 2 + n[..., 1::2] ** 2
        r2 = r[..., 0::2] ** 2 + r[..., 1::2] ** 2
    else:
        n2 = n[..., :P] ** 2 + n[..., P:] ** 2
        r2 = r[..., :P] ** 2 + r[..., P:] ** 2
    c2s2 = (cos.astype(np.float64) ** 2 + sin.astype(np.float64) ** 2)[:, None, :]
    np.testing.assert_allclose(r2, n2 * c2s2, rtol=1e-13, atol=1e-300)


def test_split_half_is_permuted_interleaved(oracle_mod):
    heads, D = 5, 16
    P = D // 2
    rows = 12
    x = _rows(24, rows, heads * D)
    w = synth.normal_bf16(24, 2, heads * D, 1.0, 0.1)
    cos, sin = synth.rope_table_3axis(2, 2, 3, D, (2, 3, 3))
    # Q maps split-half index p -> 2p and p + P -> 2p + 1 inside each head
    perm = np.empty(D, np.int64)
    perm[0::2] = np.arange(P)
    perm[1::2] = np.arange(P) + P
    full = (np.arange(heads)[:, None] * D + perm[None, :]).ravel()
    xq = x[:, full]
    wq = w[full]
    ys, es = oracle_mod.rms_norm_rope(x, w, cos, sin, heads, D, 1, 1e-6, exact=True)
    yi, ei = oracle_mod.rms_norm_rope(xq, wq, cos, sin, heads, D, 0, 1e-6, exact=True)
    inv = np.argsort(full)
    np.testing.assert_allclose(ei[:, inv], es, rtol=1e-15, atol=1e-300)
    assert np.array_equal(yi[:, inv], ys)


def test_rope_position_is_row_mod_table_rows(oracle_mod):
    # batch of 3 sequences of 4 positions: rows 4..7 and 8..11 repeat 0..3
    heads, D = 2, 8
    x = _rows(25, 4, heads * D)
    xb = np.concatenate([x, x, x])
    cos, sin = synth.rope_table_1d(4, D)
    y1 = oracle_mod.rms_norm_rope(x, None, cos, sin, heads, D, 0, 1e-6)
    yb = oracle_mod.rms_norm_rope(xb, None, cos, sin, heads, D, 0, 1e-6)
    assert np.array_equal(yb, np.concatenate([y1, y1, y1]))
    # and per-row tables with table_rows == rows give the same answer
    cb, sb = np.concatenate([cos] * 3), np.concatenate([sin] * 3)
    assert np.array_equal(
        oracle_mod.rms_norm_rope(xb, None, cb, sb, heads, D, 0, 1e-6), yb)


def test_rope_rejects_bad_arguments(oracle_mod):
    x = _rows(26, 2, 8)
    c, s = _const_tables(1, 4, 1.0, 0.0)
    with pytest.raises(RuntimeError):
        oracle_mod.rms_norm_rope(x, None, c, s, 1, 8, 2, 1e-6)


# ------------------------------------------------------------ AdaLN pins --

ADALN_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "adaln_hand_cases_h4.txt")


def _parse_adaln():
    cases = []
    for line in open(ADALN_GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, eps, xs, ws, sc, sh, rpc, exact, bits = [s.strip() for s in line.split(" | ")]
        rows = lambda t: np.array([list(map(float, r.split())) for r in t.split(";")])
        x = rows(xs)
        cases.append(dict(
            name=name, eps=float(eps), x=x,
            w=None if ws == "-" else np.array(list(map(float, ws.split()))),
            scale=rows(sc), shift=rows(sh), rows_per_cond=int(rpc),
            exact=np.array(list(map(float, exact.split()))).reshape(x.shape),
            bits=np.array([int(b, 16) for b in bits.split()], np.uint16).reshape(x.shape)))
    return cases


@pytest.mark.parametrize("case", _parse_adaln(), ids=lambda c: c["name"])
def test_adaln_hand_cases(oracle_mod, case):
    y, ye = oracle_mod.rms_norm_adaln(
        bits_of(case["x"]), None if case["w"] is None else bits_of(case["w"]),
        bits_of(case["scale"]), bits_of(case["shift"]), case["eps"],
        rows_per_cond=case["rows_per_cond"], exact=True)
    assert np.array_equal(y, case["bits"]), [hex(v) for v in y.ravel()]
    np.testing.assert_allclose(ye, case["exact"], rtol=4e-16, atol=1e-300)


def _cond(seed, n, H, lo, hi):
    return synth.uniform_bf16(seed, 3, n * H, lo, hi).reshape(n, H)


def test_adaln_zero_modulation_is_rms_norm(oracle_mod):
    x = _rows(41, 12, 96)
    w = synth.normal_bf16(41, 2, 96, 1.0, 0.1)
    zero = np.zeros((3, 96), np.uint16)
    y, ye = oracle_mod.rms_norm_adaln(x, w, zero, zero, 1e-6, rows_per_cond=4, exact=True)
    yn, yne = oracle_mod.rms_norm(x, w, 1e-6, exact=True)
    assert np.array_equal(y, yn) and np.array_equal(ye, yne)


def test_adaln_scale_minus_one_gives_shift(oracle_mod):
    x = _rows(42, 6, 40)
    shift = _cond(42, 2, 40, -3, 3)
    minus1 = bits_of(-np.ones((2, 40)))
    y = oracle_mod.rms_norm_adaln(x, None, minus1, shift, 1e-6, rows_per_cond=3)
    assert np.array_equal(y, np.repeat(shift, 3, axis=0))


def test_adaln_is_affine_in_scale_and_shift(oracle_mod):
    x = _rows(43, 8, 64)
    w = synth.normal_bf16(43, 2, 64, 1.0, 0.1)
    s = _cond(43, 2, 64, -0.5, 0.5)
    t = _cond(44, 2, 64, -2, 2)
    zero = np.zeros_like(s)
    _, n = oracle_mod.rms_norm(x, w, 1e-6, exact=True)
    _, ys = oracle_mod.rms_norm_adaln(x, w, s, zero, 1e-6, rows_per_cond=4, exact=True)
    _, yst = oracle_mod.rms_norm_adaln(x, w, s, t, 1e-6, rows_per_cond=4, exact=True)
    sw = np.repeat(oracle_mod.widen_bf16(s), 4, axis=0)
    tw = np.repeat(oracle_mod.widen_bf16(t), 4, axis=0)
    np.testing.assert_allclose(ys, n * (1 + sw), rtol=1e-15, atol=1e-300)
    np.testing.assert_allclose(yst - ys, tw, rtol=0, atol=1e-14)


def test_adaln_conditioning_rows(oracle_mod):
    # rows_per_cond consecutive rows share one conditioning row; a ragged last
    # group uses the next conditioning row
    x = _rows(45, 7, 32)
    s = _cond(45, 3, 32, -1, 1)
    t = _cond(46, 3, 32, -1, 1)
    y = oracle_mod.rms_norm_adaln(x, None, s, t, 1e-6, rows_per_cond=3)
    parts = [oracle_mod.rms_norm_adaln(x[c * 3:(c + 1) * 3], None, s[c:c + 1], t[c:c + 1],
                                       1e-6, rows_per_cond=3) for c in range(3)]
    assert np.array_equal(y, np.concatenate(parts))
    assert np.array_equal(oracle_mod.rms_norm_adaln(x, None, s, t, 1e-6, rows_per_cond=3,
                                                    threads=3), y)


# ------------------------------------------------------ residual-add pins --

def test_add_norm_hand_cases(oracle_mod):
    # h = x + res = (3, 4, 0, 0) exactly -> y = (1.2, 1.6, 0, 0) (see
    # hand_cases_h4.txt for the bf16 bits 0x3F9A, 0x3FCD)
    x = bits_of([[1, 1, -1, 2]])
    r = bits_of([[2, 3, 1, -2]])
    y, h, ye = oracle_mod.add_rms_norm(x, r, None, 0.0, exact=True)
    assert h.ravel().tolist() == [0x4040, 0x4080, 0x0000, 0x0000]     # 3, 4, 0, 0
    assert y.ravel().tolist() == [0x3F9A, 0x3FCD, 0x0000, 0x0000]
    np.testing.assert_allclose(ye.ravel(), [1.2, 1.6, 0, 0], rtol=4e-16)
    # rounding of h, round to nearest even: 1 + 2^-8 is a tie -> 1.0 (even);
    # 1 + 3*2^-8 is a tie between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    x = bits_of([[1, 1, 1, 1]])
    r = bits_of([[2.0 ** -8, 3 * 2.0 ** -8, 0, 0]])
    y, h, ye = oracle_mod.add_rms_norm(x, r, None, 0.0, exact=True)
    assert h.ravel().tolist() == [0x3F80, 0x3F82, 0x3F80, 0x3F80]
    # the norm reads the ROUNDED h: mean = (1 + (1 + 2^-6)^2 + 1 + 1) / 4
    hv = np.array([1.0, 1 + 2.0 ** -6, 1.0, 1.0])
    np.testing.assert_allclose(ye.ravel(), hv / np.sqrt(np.mean(hv ** 2)), rtol=4e-16)


def test_add_norm_zero_residual_is_rms_norm(oracle_mod):
    x = _rows(61, 9, 96)
    w = synth.normal_bf16(61, 2, 96, 1.0, 0.1)
    zero = np.zeros_like(x)
    y, h, ye = oracle_mod.add_rms_norm(x, zero, w, 1e-6, exact=True)
    yn, yne = oracle_mod.rms_norm(x, w, 1e-6, exact=True)
    assert np.array_equal(h, x) and np.array_equal(y, yn) and np.array_equal(ye, yne)


def test_add_norm_commutes_and_cancels(oracle_mod):
    x = _rows(62, 7, 40)
    r = _rows(63, 7, 40)
    a = oracle_mod.add_rms_norm(x, r, None, 1e-6)
    b = oracle_mod.add_rms_norm(r, x, None, 1e-6)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # x + (-x) = 0 exactly: h is all zero, and with eps > 0 so is y
    neg = (x ^ np.uint16(0x8000)).astype(np.uint16)
    y, h = oracle_mod.add_rms_norm(x, neg, None, 1e-6)
    assert np.all(oracle_mod.widen_bf16(h) == 0) and np.all(oracle_mod.widen_bf16(y) == 0)


def test_add_norm_h_is_the_rounded_sum(oracle_mod):
    x = _rows(64, 16, 128)
    r = _rows(65, 16, 128, "uniform")
    _, h = oracle_mod.add_rms_norm(x, r, None, 1e-6, threads=3)
    s = oracle_mod.widen_bf16(x) + oracle_mod.widen_bf16(r)   # exact in binary64
    assert np.array_equal(h, oracle_mod.round_bf16(s))
    # and y is the RMSNorm of that h
    y, _ = oracle_mod.add_rms_norm(x, r, None, 1e-6)
    assert np.array_equal(y, oracle_mod.rms_norm(h, None, 1e-6))


# ------------------------------------------------------- GELU / GEGLU pins --

def _bf16_grid(lo, hi, n):
    v = np.linspace(lo, hi, n).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)    # truncate to bf16


def test_gelu_is_x_sigma_identity(oracle_mod):
    # z is odd in x and sigma(2z) + sigma(-2z) = 1, so gelu(x) - gelu(-x) = x
    x = _bf16_grid(0.01, 12, 3001)
    neg = (x | np.uint16(0x8000)).astype(np.uint16)
    _, gp = oracle_mod.gelu_tanh(x, exact=True)
    _, gn = oracle_mod.gelu_tanh(neg, exact=True)
    xv = oracle_mod.widen_bf16(x)
    np.testing.assert_allclose(gp - gn, xv, rtol=1e-15, atol=0)


def test_gelu_matches_tanh_form_and_torch(oracle_mod):
    # on [-2, 4] the literal tanh form is itself accurate (1 + tanh(z) >= 0.04,
    # so its cancellation costs under 3e-15); further left it is not, which is
    # why the oracle uses the sigmoid identity
    x = _bf16_grid(-2, 4, 8001)
    _, g = oracle_mod.gelu_tanh(x, exact=True)
    xv = oracle_mod.widen_bf16(x)
    z = np.sqrt(2 / np.pi) * (xv + 0.044715 * xv ** 3)
    np.testing.assert_allclose(g, 0.5 * xv * (1 + np.tanh(z)), rtol=1e-14, atol=1e-300)
    torch = pytest.importorskip("torch")
    ref = torch.nn.functional.gelu(torch.from_numpy(xv), approximate="tanh").numpy()
    np.testing.assert_allclose(g, ref, rtol=1e-14, atol=1e-300)


def test_gelu_tails(oracle_mod):
    # large x: gelu(x) = x to far below bf16 resolution
    x = _bf16_grid(6, 100, 500)
    assert np.array_equal(oracle_mod.gelu_tanh(x), x)
    # very negative x: gelu(x) = x e^{2z} / (1 + e^{2z}), so
    # log(gelu/x) = 2z - log1p(e^{2z}) -- accurate where 1 + tanh(z) cancels
    x = _bf16_grid(-11, -6, 500)
    _, g = oracle_mod.gelu_tanh(x, exact=True)
    xv = oracle_mod.widen_bf16(x)
    z = np.sqrt(2 / np.pi) * (xv + 0.044715 * xv ** 3)
    np.testing.assert_allclose(np.log(g / xv), 2 * z - np.log1p(np.exp(2 * z)), rtol=1e-13)
    assert np.all(g < 0) and np.all(g > -1e-8)
    assert int(oracle_mod.gelu_tanh(np.array([0x0000], np.uint16))[0]) == 0


def test_geglu_value_times_gelu_of_gate(oracle_mod):
    rows, h = 6, 40
    x = _rows(81, rows, 2 * h)
    y, ye = oracle_mod.geglu(x, exact=True)
    _, gate = oracle_mod.gelu_tanh(x[:, h:], exact=True)
    np.testing.assert_allclose(ye, oracle_mod.widen_bf16(x[:, :h]) * gate, rtol=1e-15,
                               atol=1e-300)
    # the halves are not interchangeable
    swapped = np.concatenate([x[:, h:], x[:, :h]], axis=1)
    assert not np.array_equal(oracle_mod.geglu(swapped), y)
    # gate -> +inf side: gelu(gate) = gate, so y = round(value * gate)
    big = np.concatenate([x[:, :h], bits_of(np.full((rows, h), 16.0))], axis=1)
    np.testing.assert_array_equal(oracle_mod.geglu(big),
                                  oracle_mod.round_bf16(oracle_mod.widen_bf16(x[:, :h]) * 16))


# ---- the other two precision modes ("cuda-kernels" page, "Supported Data
# Types": __half, __nv_bfloat16 and float) --------------------------------

ALL16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def test_f16_widen_all_patterns(oracle_mod):
    """Every binary16 pattern decodes to numpy's own binary16 value."""
    h = ALL16.view(np.float16)
    got = oracle_mod.widen(h)
    ref = h.astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_f16_round_identity_and_midpoints(oracle_mod):
    h = ALL16.view(np.float16)
    fin = np.isfinite(h)
    back = oracle_mod.round_to(h[fin].astype(np.float64), np.float16).view(np.uint16)
    assert np.array_equal(back, ALL16[fin])
    # the midpoint of two neighbours (exact in binary64) goes to the even one;
    # a hair either side goes to the nearer one
    pos = np.arange(0, 0x7C00, dtype=np.uint16)
    lo = pos[:-1].view(np.float16).astype(np.float64)
    hi = pos[1:].view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2
    even = np.where(pos[:-1] % 2 == 0, pos[:-1], pos[1:])
    assert np.array_equal(oracle_mod.round_to(mid, np.float16).view(np.uint16), even)
    assert np.array_equal(oracle_mod.round_to(-mid, np.float16).view(np.uint16), even | 0x8000)
    eps = (hi - lo) * 2.0 ** -20
    assert np.array_equal(oracle_mod.round_to(mid - eps, np.float16).view(np.uint16), pos[:-1])
    assert np.array_equal(oracle_mod.round_to(mid + eps, np.float16).view(np.uint16), pos[1:])


def test_f16_round_specials(oracle_mod):
    v = np.array([65504.0, 65519.99, 65520.0, -65520.0, 1e300, np.inf, -np.inf, 0.0, -0.0,
                  2.0 ** -25, 2.0 ** -25 * 1.0001, 2.0 ** -24, 3 * 2.0 ** -26, 2.0 ** -14])
    got = oracle_mod.round_to(v, np.float16).view(np.uint16)
    assert list(got) == [0x7BFF, 0x7BFF, 0x7C00, 0xFC00, 0x7C00, 0x7C00, 0xFC00, 0x0000, 0x8000,
                         0x0000, 0x0001, 0x0001, 0x0001, 0x0400]
    assert np.isnan(oracle_mod.round_to(np.array([np.nan]), np.float16)[0])


def test_f16_round_matches_numpy_conversion(oracle_mod):
    """numpy converts binary64 to binary16 with its own round-to-nearest-even."""
    rng = np.random.default_rng(3)
    v = rng.standard_normal(200000) * np.exp2(rng.uniform(-30, 17, 200000))
    got = oracle_mod.round_to(v, np.float16)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


def test_f32_round_matches_hardware_conversion(oracle_mod):
    """The host's binary64 -> binary32 conversion (round to nearest even) is
    an independent implementation of the same rounding."""
    rng = np.random.default_rng(4)
    v = rng.standard_normal(200000) * np.exp2(rng.uniform(-155, 130, 200000))
    # exact midpoints between binary32 neighbours, subnormal ones included
    f = (rng.integers(1, 0x7F7FFFFF, 100000, dtype=np.uint64).astype(np.uint32)).view(np.float32)
    nxt = np.nextafter(f, np.float32(np.inf))
    mids = (f.astype(np.float64) + nxt.astype(np.float64)) / 2
    for vals in (v, mids, -mids):
        got = oracle_mod.round_to(vals, np.float32)
        with np.errstate(over="ignore"):
            ref = vals.astype(np.float32)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    big = np.float64(np.finfo(np.float32).max)
    half_ulp = 2.0 ** 103
    got = oracle_mod.round_to(np.array([big + half_ulp * 0.999, big + half_ulp]), np.float32)
    assert got[0] == np.finfo(np.float32).max and np.isinf(got[1])


def _shared_values(seed, rows, H):
    """Values exactly representable in bf16, binary16 and binary32: 8
    significant bits, magnitudes within binary16's normal range."""
    x = synth.uniform_bf16(seed, 0, rows * H, -4.0, 4.0).reshape(rows, H)
    xf = synth.bf16_bits_to_f32(x)
    xf = np.where(np.abs(xf) < 2.0 ** -13, 0.0, xf).astype(np.float32)
    return synth.to_bf16_bits(xf), xf


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_formats_share_the_arithmetic(oracle_mod, dtype):
    """Inputs that every format holds exactly give the same exact results in
    every format, and each output is that format's rounding of them."""
    xb, xf = _shared_values(21, 6, 32)
    wb, wf = _shared_values(22, 1, 32)
    wb, wf = wb[0], wf[0]
    cast = (lambda a: a.astype(dtype))
    _, e_b = oracle_mod.rms_norm(xb, wb, 1e-6, exact=True)
    y, e = oracle_mod.rms_norm(cast(xf), cast(wf), 1e-6, exact=True)
    bits = (lambda a: a.view(np.uint16 if dtype == np.float16 else np.uint32))
    assert y.dtype == dtype and np.array_equal(e, e_b)
    assert np.array_equal(bits(y), bits(oracle_mod.round_to(e, dtype)))
    c, s = synth.rope_table_1d(6, 8)
    for mode in (0, 1):
        _, e_b = oracle_mod.rms_norm_rope(xb, wb, c, s, 4, 8, mode, 1e-6, exact=True)
        y, e = oracle_mod.rms_norm_rope(cast(xf), cast(wf), c, s, 4, 8, mode, 1e-6, exact=True)
        assert np.array_equal(e, e_b) and np.array_equal(bits(y), bits(oracle_mod.round_to(e, dtype)))
    sb, sf = _shared_values(23, 2, 32)
    tb, tf = _shared_values(24, 2, 32)
    _, e_b = oracle_mod.rms_norm_adaln(xb, wb, sb, tb, 1e-6, rows_per_cond=3, exact=True)
    y, e = oracle_mod.rms_norm_adaln(cast(xf), cast(wf), cast(sf), cast(tf), 1e-6,
                                     rows_per_cond=3, exact=True)
    assert np.array_equal(e, e_b) and np.array_equal(bits(y), bits(oracle_mod.round_to(e, dtype)))
    rb, rf = _shared_values(25, 6, 32)
    y, h, e = oracle_mod.add_rms_norm(cast(xf), cast(rf), cast(wf), 1e-6, exact=True)
    assert np.array_equal(bits(h), bits(oracle_mod.round_to(xf.astype(np.float64) + rf, dtype)))
    _, e_h = oracle_mod.rms_norm(h, cast(wf), 1e-6, exact=True)
    assert np.array_equal(e, e_h) and np.array_equal(bits(y), bits(oracle_mod.round_to(e, dtype)))
    _, e_b = oracle_mod.gelu_tanh(xb, exact=True)
    y, e = oracle_mod.gelu_tanh(cast(xf), exact=True)
    assert y.dtype == dtype and np.array_equal(e, e_b)
    assert np.array_equal(bits(y), bits(oracle_mod.round_to(e, dtype)))
    _, e_b = oracle_mod.geglu(xb, exact=True)
    y, e = oracle_mod.geglu(cast(xf), exact=True)
    assert y.dtype == dtype and y.shape == (6, 16) and np.array_equal(e, e_b)
    assert np.array_equal(bits(y), bits(oracle_mod.round_to(e, dtype)))


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_formats_match_torch_rms_norm_fp64(oracle_mod, dtype):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    if not hasattr(F, "rms_norm"):
        pytest.skip("torch without rms_norm")
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((8, 3072)) * 3).astype(dtype)
    w = (1 + 0.1 * rng.standard_normal(3072)).astype(dtype)
    _, ye = oracle_mod.rms_norm(x, w, 1e-6, exact=True)
    ref = F.rms_norm(torch.from_numpy(x.astype(np.float64)), (3072,),
                     torch.from_numpy(w.astype(np.float64)),
                     eps=float(np.float32(1e-6))).numpy()
    np.testing.assert_allclose(ye, ref, rtol=1e-12, atol=1e-300)


def _f32_grid(lo, hi, n, seed):
    """n float32 values in [lo, hi] with full 24-bit significands."""
    rng = np.random.default_rng(seed)
    return rng.uniform(lo, hi, n).astype(np.float32)


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_gelu_formats_match_torch_and_numpy_rounding(oracle_mod, dtype):
    # [-2, 4]: the literal tanh form is accurate there (see the bf16 pin), and
    # torch's fp64 GELU gives the exact value; the stored result is numpy's
    # own round-to-nearest-even conversion of it
    torch = pytest.importorskip("torch")
    if dtype == np.float16:
        x = ALL16.view(np.float16)
        x = x[np.isfinite(x) & (x >= -2) & (x <= 4)]
    else:
        x = _f32_grid(-2, 4, 20001, 31)
    y, g = oracle_mod.gelu_tanh(x, exact=True)
    ref = torch.nn.functional.gelu(torch.from_numpy(x.astype(np.float64)),
                                   approximate="tanh").numpy()
    np.testing.assert_allclose(g, ref, rtol=1e-14, atol=1e-300)
    assert y.dtype == dtype and np.array_equal(y, g.astype(dtype))


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_gelu_formats_tails_and_specials(oracle_mod, dtype):
    lim = 60000.0 if dtype == np.float16 else 1e30
    big = np.array([6, 9.5, 100, 1000, lim], dtype)
    assert np.array_equal(oracle_mod.gelu_tanh(big), big)          # gelu(x) = x
    # left tail: log(gelu/x) = 2z - log1p(e^{2z}), accurate where 1 + tanh z cancels
    x = (np.linspace(-6, -1, 400) if dtype == np.float16 else _f32_grid(-20, -6, 400, 32)).astype(dtype)
    y, g = oracle_mod.gelu_tanh(x, exact=True)
    xv = x.astype(np.float64)
    z = np.sqrt(2 / np.pi) * (xv + 0.044715 * xv ** 3)
    np.testing.assert_allclose(np.log(g / xv), 2 * z - np.log1p(np.exp(2 * z)), rtol=1e-13)
    assert np.array_equal(y, g.astype(dtype))        # down into the subnormals and zero
    inf = np.array([np.inf, -np.inf, np.nan, -lim, 0.0, -0.0], dtype)
    y = oracle_mod.gelu_tanh(inf)
    assert y[0] == np.inf and np.isnan(y[1]) and np.isnan(y[2])   # -inf * 0 is NaN
    assert y[3] == 0 and np.signbit(y[3]) and y[4] == 0 and not np.signbit(y[4])
    assert np.signbit(y[5])


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_geglu_formats_value_times_gelu_of_gate(oracle_mod, dtype):
    rng = np.random.default_rng(33)
    rows, h = 5, 24
    x = (rng.standard_normal((rows, 2 * h)) * 3).astype(dtype)
    if dtype == np.float32:
        # huge values on far-tail gates: the product is normal although the
        # gelu of the gate is below binary32's smallest normal number
        x[0, :h] = np.float32(2.0 ** 120)
        x[0, h:] = np.linspace(-11.5, -10.5, h).astype(np.float32)
    y, ye = oracle_mod.geglu(x, exact=True)
    _, gate = oracle_mod.gelu_tanh(np.ascontiguousarray(x[:, h:]), exact=True)
    np.testing.assert_allclose(ye, x[:, :h].astype(np.float64) * gate, rtol=1e-15, atol=1e-300)
    assert y.dtype == dtype and np.array_equal(y, ye.astype(dtype))
    if dtype == np.float32:
        assert np.all(np.abs(gate[0]) < 2.0 ** -126) and np.all(np.abs(y[0]) > 2.0 ** -100)
    swapped = np.concatenate([x[:, h:], x[:, :h]], axis=1)
    assert not np.array_equal(oracle_mod.geglu(swapped), y)


def test_formats_reject_mixed_dtypes(oracle_mod):
    x = np.zeros((2, 8), np.float16)
    with pytest.raises(TypeError):
        oracle_mod.rms_norm(x, np.ones(8, np.float32), 1e-6)
    with pytest.raises(TypeError):
        oracle_mod.rms_norm(x.astype(np.float64), None, 1e-6)


# ---- standalone RoPE with angles from token positions ("Kernel-Specific
# Guidelines / RoPE": 1D [batch, seq, heads, head_dim], 3D [batch, t*h*w,
# heads, head_dim]) ----------------------------------------------------------

def _unit_pairs(rows, heads, D, mode, which):
    """Rows whose every rotation pair is (1, 0) (which=0) or (0, 1) (which=1),
    as float32 (exact in every format)."""
    x = np.zeros((rows, heads, D), np.float32)
    P = D // 2
    if mode == 0:
        x[:, :, which::2] = 1.0
    else:
        x[:, :, which * P:(which + 1) * P] = 1.0
    return x.reshape(rows, heads * D)


def _pair(ye, heads, D, mode, p):
    """(first, second) element of pair p of head 0 of every row."""
    P = D // 2
    ia, ib = (2 * p, 2 * p + 1) if mode == 0 else (p, p + P)
    return ye[:, ia], ye[:, ib]


def test_rope_positions_identity_at_token_zero(oracle_mod):
    x = synth.normal_bf16(90, 0, 3 * 4 * 16).reshape(3, 64)
    for mode in (0, 1):
        y = oracle_mod.rope(x, 4, 16, mode, (1, 1, 1), (8, 0, 0))
        assert np.array_equal(y, x)


@pytest.mark.parametrize("mode", [0, 1])
def test_rope_positions_closed_form_frequencies(oracle_mod, mode):
    """1D, head_dim 128, theta 1e4: pair k turns by position * 1e4^(-k/64);
    pair 32 by position/100 and pair 16 by position/10 (exact in reals), and
    pair 0 by the position itself.  Row 100 is position 100."""
    import math
    D = 128
    for which in (0, 1):
        x = _unit_pairs(101, 1, D, mode, which)
        _, ye = oracle_mod.rope(x, 1, D, mode, (4096, 1, 1), (64, 0, 0), 10000.0, exact=True)
        for p, ang in ((32, 1.0), (16, 10.0), (0, 100.0)):
            a, b = _pair(ye, 1, D, mode, p)
            if which == 0:   # (1, 0) -> (cos, sin)
                assert abs(a[100] - math.cos(ang)) < 1e-13 and abs(b[100] - math.sin(ang)) < 1e-13
            else:            # (0, 1) -> (-sin, cos)
                assert abs(a[100] + math.sin(ang)) < 1e-13 and abs(b[100] - math.cos(ang)) < 1e-13


def test_rope_positions_three_axis_coordinates(oracle_mod):
    """Grid (3, 4, 5), pairs (2, 3, 3): token (1*4 + 2)*5 + 3 = 33 has
    coordinates (1, 2, 3); the first pair of each axis turns by the
    coordinate, the second pair of the two-pair t axis by 1e4^(-1/2) = 0.01."""
    import math
    D = 16
    x = _unit_pairs(34, 1, D, 0, 0)
    _, ye = oracle_mod.rope(x, 1, D, 0, (3, 4, 5), (2, 3, 3), 10000.0, exact=True)
    for p, ang in ((0, 1.0), (2, 2.0), (5, 3.0), (1, 0.01)):
        a, b = _pair(ye, 1, D, 0, p)
        assert abs(a[33] - math.cos(ang)) < 1e-13 and abs(b[33] - math.sin(ang)) < 1e-13


def test_rope_positions_angle_is_additive_in_position(oracle_mod):
    """cos(t(p+q)) = cos(tp)cos(tq) - sin(tp)sin(tq) for every pair: the angle
    is linear in the position, with no offset."""
    D = 32
    x = _unit_pairs(40, 1, D, 0, 0)
    _, ye = oracle_mod.rope(x, 1, D, 0, (64, 1, 1), (16, 0, 0), 500.0, exact=True)
    c, s = ye[:, 0::2], ye[:, 1::2]
    for p, q in ((3, 5), (7, 11), (0, 13), (19, 20)):
        assert np.allclose(c[p + q], c[p] * c[q] - s[p] * s[q], atol=1e-12)
        assert np.allclose(s[p + q], s[p] * c[q] + c[p] * s[q], atol=1e-12)


def test_rope_positions_norms_wrap_and_permutation(oracle_mod):
    heads, D = 3, 12
    x = synth.normal_bf16(91, 0, 50 * heads * D).reshape(50, heads * D)
    grid, pairs = (2, 3, 4), (2, 2, 2)
    y0, e0 = oracle_mod.rope(x, heads, D, 0, grid, pairs, exact=True)
    xw = oracle_mod.widen_bf16(x).reshape(50, heads, D // 2, 2)
    ew = e0.reshape(50, heads, D // 2, 2)
    assert np.allclose(np.hypot(ew[..., 0], ew[..., 1]), np.hypot(xw[..., 0], xw[..., 1]),
                       rtol=1e-14, atol=1e-300)
    # row r and row r + 24 are the same token
    y1 = oracle_mod.rope(np.concatenate([x[24:48], x[:24]]), heads, D, 0, grid, pairs)
    assert np.array_equal(y1[:24], y0[24:48]) and np.array_equal(y1[24:48], y0[:24])
    # row blocks on several threads keep their tokens
    assert np.array_equal(oracle_mod.rope(x, heads, D, 0, grid, pairs, threads=4), y0)
    # split-half is interleaved under the pair permutation
    perm = np.concatenate([np.arange(0, D, 2), np.arange(1, D, 2)])
    xs = x.reshape(50, heads, D)[:, :, perm].reshape(50, heads * D)
    ys = oracle_mod.rope(xs, heads, D, 1, grid, pairs)
    assert np.array_equal(ys.reshape(50, heads, D)[:, :, np.argsort(perm)].reshape(50, -1), y0)


def test_rope_positions_rejects_bad_arguments(oracle_mod):
    x = np.zeros((2, 16), np.uint16)
    for grid, pairs, theta in (((2, 1, 1), (3, 0, 0), 1e4), ((0, 1, 1), (4, 0, 0), 1e4),
                               ((2, 1, 1), (4, 0, 0), 0.0), ((2, 1, 1), (5, -1, 0), 1e4)):
        with pytest.raises(RuntimeError):
            oracle_mod.rope(x, 2, 8, 0, grid, pairs, theta)


def test_rope_tables_are_the_fused_forms_table_recipe(oracle_mod):
    """The positional angles, written as tables, are the tables the fused
    form's workloads are generated with (the generator's own fp64 code, cast
    to fp32): the standalone and fused RoPE agree on what a position means."""
    c, s = oracle_mod.rope_tables(6144, 64, (8, 24, 32), (10, 11, 11))
    ct, st = synth.rope_table_3axis(8, 24, 32, 64, (10, 11, 11), 10000.0)
    assert np.abs(c - ct).max() <= 2.0 ** -24 and np.abs(s - st).max() <= 2.0 ** -24
    c, s = oracle_mod.rope_tables(4096, 128, (4096, 1, 1), (64, 0, 0))
    ct, st = synth.rope_table_1d(4096, 128)
    assert np.abs(c - ct).max() <= 2.0 ** -24 and np.abs(s - st).max() <= 2.0 ** -24


def test_rope_tables_identity_wrap_and_norms(oracle_mod):
    c, s = oracle_mod.rope_tables(2 * 96 + 5, 64, (2, 6, 8), (10, 11, 11))
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)                 # token 0: no turn
    assert np.array_equal(c[:96 + 5], c[96:2 * 96 + 5])                # row s is token s mod THW
    np.testing.assert_allclose(c * c + s * s, 1.0, rtol=1e-15)
    with pytest.raises(ValueError):
        oracle_mod.rope_tables(4, 64, (2, 6, 8), (10, 11, 10))          # pairs must sum to D/2
