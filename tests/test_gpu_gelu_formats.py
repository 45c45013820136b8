"""GPU parity of the tanh-approximated GELU and of GEGLU in fp16 and fp32
("cuda-kernels" skill page, "Supported Data Types": __half and float beside
__nv_bfloat16; "Kernel-Specific Guidelines / GEGLU vs GELU") against the
fp64 oracle, element by element.

fp16: at most 1 ulp (ordinal distance; NaN matches NaN), on every fp16 input
for GELU and every fp16 gate for GEGLU.  fp32: the bound of
oracle.compare.gelu_f32_bound (fp32 rounding of q magnified by 2^q in the
left tail, the ex2/rcp approximations, one rounding into the subnormals),
on random bit patterns of every exponent, a dense grid of the active range,
the specials, and huge values times far-tail gates (the exact path).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import rope_element_dit_gb300 as L
import synth
from oracle.compare import compare_fmt, compare_fmt_bounded, gelu_f32_bound

pytestmark = pytest.mark.gpu

THREADS = min(32, os.cpu_count() or 1)
GUARD = 64
CODES = {np.float16: L.DTYPE_F16, np.float32: L.DTYPE_F32}
CANARY = {np.float16: np.uint16(0x7E01), np.float32: np.uint32(0x7FC00001)}
UINT = {np.float16: np.uint16, np.float32: np.uint32}
TORCH = {np.float16: torch.float16, np.float32: torch.float32}


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU parity tests need a CUDA device"
    torch.cuda.set_device(0)
    assert torch.cuda.get_device_capability(0) == (10, 3)


def stream():
    return torch.cuda.current_stream().cuda_stream


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def guarded(n, dtype):
    """An n-element output inside canary words on both sides."""
    c = np.full(n + 2 * GUARD, CANARY[dtype], UINT[dtype]).view(dtype)
    whole = to_dev(c)
    return whole, whole[GUARD:GUARD + n]


def check_guard(whole, n, dtype):
    h = whole.cpu().numpy().view(UINT[dtype])
    assert np.all(h[:GUARD] == CANARY[dtype]) and np.all(h[GUARD + n:] == CANARY[dtype]), \
        "kernel wrote outside its output"


def gpu_gelu(xd, n, out, dtype):
    st = L.ltxk_gelu_tanh_dt(out.data_ptr(), xd.data_ptr(), n, CODES[dtype], stream())
    assert st == L.OK, L.ltxk_status_string(st)


def gpu_geglu(xd, rows, hidden, out, dtype):
    st = L.ltxk_geglu_dt(out.data_ptr(), xd.data_ptr(), rows, hidden, CODES[dtype], stream())
    assert st == L.OK, L.ltxk_status_string(st)


def assert_gelu_parity(got, x, what, gate=None, exact=None, chunk=1 << 24):
    """fp16: 1 ulp against the oracle's rounding; fp32: the derived bound.
    ``gate``/``exact``: the fp32 bound's inputs (default: x and GELU's exact
    values)."""
    got = np.asarray(got).reshape(-1)
    if got.dtype == np.float16:
        ref = oracle.gelu_tanh(x) if exact is None else oracle.round_to(exact, np.float16)
        for s in range(0, got.size, chunk):
            r = compare_fmt(got[s:s + chunk], np.asarray(ref).reshape(-1)[s:s + chunk])
            assert r["ok"], f"{what}[{s}:]: {r}"
        return
    if exact is None:
        _, exact = oracle.gelu_tanh(x, exact=True, threads=THREADS)
    gate = np.asarray(x if gate is None else gate).reshape(-1)
    exact = np.asarray(exact).reshape(-1)
    for s in range(0, got.size, chunk):
        e = exact[s:s + chunk]
        r = compare_fmt_bounded(got[s:s + chunk], e, gelu_f32_bound(gate[s:s + chunk], e))
        assert r["ok"], f"{what}[{s}:]: {r}"


def f32_inputs(seed, n_random=1 << 21, n_grid=1 << 20):
    """Random bit patterns over every exponent (NaN, infinities and
    subnormals included), a dense grid of [-13, 13], and the specials."""
    rng = np.random.default_rng(seed)
    rand = rng.integers(0, 1 << 32, n_random, dtype=np.uint64).astype(np.uint32).view(np.float32)
    grid = np.linspace(-13, 13, n_grid).astype(np.float32)
    spec = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45, 1.17549435e-38,
                     3.4028235e38, -3.4028235e38, 1e30, -1e30, 10.3, -10.3, -64.0],
                    np.float32)
    return np.concatenate([rand, grid, spec])


F16_ALL = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)


# -------------------------------------------------------------------- GELU --

@pytest.mark.parametrize("offset", [0, 1, 3])
def test_gelu_f16_every_value(offset):
    """All 65536 fp16 inputs; offset 1 and 3 take the element kernel."""
    n = F16_ALL.size
    xd = to_dev(np.concatenate([np.zeros(offset, np.float16), F16_ALL]))
    whole, out = guarded(n + offset, np.float16)
    gpu_gelu(xd[offset:], n, out[offset:], np.float16)
    torch.cuda.synchronize()
    check_guard(whole, n + offset, np.float16)
    assert_gelu_parity(out[offset:].cpu().numpy(), F16_ALL, f"offset {offset}")


@pytest.mark.parametrize("offset", [0, 1])
def test_gelu_f32_values(offset):
    x = f32_inputs(71 + offset)
    n = x.size
    xd = to_dev(np.concatenate([np.zeros(offset, np.float32), x]))
    whole, out = guarded(n + offset, np.float32)
    gpu_gelu(xd[offset:], n, out[offset:], np.float32)
    torch.cuda.synchronize()
    check_guard(whole, n + offset, np.float32)
    assert_gelu_parity(out[offset:].cpu().numpy(), x, f"offset {offset}")


def test_gelu_f32_core_is_tighter_than_the_bound():
    """On [-6, 6] the fp32 result meets the bound with k0 = 16 instead of 32:
    no accuracy is given away where the function is well conditioned (a q
    offset by 64 before ex2 would cost ~2^-18 = 64 units at q = 0)."""
    x = np.linspace(-6, 6, 1 << 20).astype(np.float32)
    out = torch.empty(x.size, dtype=torch.float32, device="cuda")
    gpu_gelu(to_dev(x), x.size, out, np.float32)
    torch.cuda.synchronize()
    _, e = oracle.gelu_tanh(x, exact=True)
    g = out.cpu().numpy().astype(np.float64)
    err = np.abs(g - e)
    tight = gelu_f32_bound(x, e, k0=16.0)
    assert np.all(err <= tight), float(np.max(err / tight))


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 4097, 65543, 1000003])
def test_gelu_formats_ragged_sizes(dtype, n):
    x = synth.normal_with_outliers_bf16(2100 + n, n, 0.01, 50.0, fmt="f16" if dtype == np.float16
                                        else "f32")
    whole, out = guarded(n, dtype)
    gpu_gelu(to_dev(x), n, out, dtype)
    torch.cuda.synchronize()
    check_guard(whole, n, dtype)
    assert_gelu_parity(out.cpu().numpy(), x, f"n={n}")


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_gelu_formats_in_place_and_helper(dtype):
    n = 4096 * 3 + 5
    x = synth.uniform_bf16(33, 0, n, -12.0, 6.0, fmt="f16" if dtype == np.float16 else "f32")
    xd = to_dev(x)
    gpu_gelu(xd, n, xd, dtype)
    torch.cuda.synchronize()
    assert_gelu_parity(xd.cpu().numpy(), x, "in place")
    t = to_dev(x[:3 * 5 * 800]).reshape(3, 5, 800)
    y = L.gelu_tanh(t)
    torch.cuda.synchronize()
    assert y.shape == t.shape and y.dtype == TORCH[dtype]
    assert_gelu_parity(y.cpu().numpy(), x[:3 * 5 * 800], "helper")
    assert L.ltxk_gelu_tanh_dt(xd.data_ptr(), xd.data_ptr(), 0, CODES[dtype], stream()) == L.OK


@pytest.mark.parametrize("name", ["gelu_f16", "gelu_f32"])
def test_gelu_formats_workload_full_size(name):
    case = synth.WORKLOADS[name][0]
    dtype = synth.FORMATS[case.dtype]
    x = synth.make_x(case)
    n = x.size
    whole, out = guarded(n, dtype)
    gpu_gelu(to_dev(x), n, out, dtype)
    torch.cuda.synchronize()
    check_guard(whole, n, dtype)
    if dtype == np.float16:
        got = out.cpu().numpy()
        r = compare_fmt(got, oracle.gelu_tanh(x, threads=THREADS))
        assert r["ok"], r
    else:
        assert_gelu_parity(out.cpu().numpy(), x, case.name)


# ------------------------------------------------------------------- GEGLU --

def assert_geglu_parity(got, x, what):
    h = x.shape[-1] // 2
    y, ye = oracle.geglu(x, exact=True, threads=THREADS)
    got = np.asarray(got).reshape(y.shape)
    if got.dtype == np.float16:
        r = compare_fmt(got, y)
        assert r["ok"], f"{what}: {r}"
    else:
        gate = np.ascontiguousarray(x[..., h:])
        assert_gelu_parity(got, None, what, gate=gate, exact=ye)


def wide_f16_values(seed, n):
    """fp16 values of random sign, log2-magnitude uniform in [-24, 15.9]."""
    rng = np.random.default_rng(seed)
    v = np.exp2(rng.uniform(-24, 15.9, n)) * rng.choice([-1.0, 1.0], n)
    return v.astype(np.float16)


def test_geglu_f16_every_gate_value():
    """Every fp16 gate once, against values spread over fp16's range."""
    rows, hidden = 256, 256
    g = F16_ALL.reshape(rows, hidden)
    v = wide_f16_values(81, F16_ALL.size).reshape(rows, hidden)
    x = np.concatenate([v, g], axis=1)
    whole, out = guarded(rows * hidden, np.float16)
    gpu_geglu(to_dev(x), rows, hidden, out, np.float16)
    torch.cuda.synchronize()
    check_guard(whole, rows * hidden, np.float16)
    assert_geglu_parity(out.cpu().numpy(), x, "every gate")


@pytest.mark.parametrize("rows,hidden", [(512, 4096), (3, 4097)])
def test_geglu_f32_gates_and_deep_tail(rows, hidden):
    """fp32 gates over every exponent and the active range, against values
    of magnitude 2^-126 .. 2^127; a band of rows pairs huge values with
    gates whose gelu is below the smallest normal (the exact path)."""
    rng = np.random.default_rng(82 + hidden)
    n = rows * hidden
    g = f32_inputs(83, n_random=n // 2, n_grid=n - n // 2 - 15)[:n].reshape(rows, hidden)
    v = (np.exp2(rng.uniform(-126, 127, n)) * rng.choice([-1.0, 1.0], n)).astype(np.float32)
    v = v.reshape(rows, hidden)
    band = slice(0, max(1, rows // 4))
    g[band] = rng.uniform(-11.8, -10.0, g[band].shape).astype(np.float32)
    v[band] = (np.exp2(rng.uniform(100, 127, v[band].shape)) *
               rng.choice([-1.0, 1.0], v[band].shape)).astype(np.float32)
    x = np.concatenate([v, g], axis=1)
    whole, out = guarded(n, np.float32)
    gpu_geglu(to_dev(x), rows, hidden, out, np.float32)
    torch.cuda.synchronize()
    check_guard(whole, n, np.float32)
    assert_geglu_parity(out.cpu().numpy(), x, f"{rows}x{hidden}")
    # the band's results are normal numbers although gelu(gate) is not
    y = out.cpu().numpy().reshape(rows, hidden)[band]
    assert np.all((np.abs(y) > 2.0 ** -126) | (y == 0))


def test_geglu_f32_tiny_gates_under_huge_values():
    """Subnormal and tiny gates (gelu(g) ~ g/2) under values of 2^100 ..
    2^127: the products are normal numbers, and the kernel must not round
    gelu(g) into the subnormals before the value scales it up."""
    rng = np.random.default_rng(84)
    rows, hidden = 64, 1024
    n = rows * hidden
    mag = np.exp2(rng.uniform(-149, -100, n))
    g = (mag * rng.choice([-1.0, 1.0], n)).astype(np.float32).reshape(rows, hidden)
    v = (np.exp2(rng.uniform(100, 127, n)) * rng.choice([-1.0, 1.0], n)).astype(np.float32)
    x = np.concatenate([v.reshape(rows, hidden), g], axis=1)
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    gpu_geglu(to_dev(x), rows, hidden, out, np.float32)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.count_nonzero(np.abs(got) > 2.0 ** -126) > n // 2
    assert_geglu_parity(got, x, "tiny gates")


# (11, 12) and (7, 1004): hidden % 4 == 0 but not % 8 -- the fp32 chunk
# kernel, the 16-bit element kernel
GEGLU_SHAPES = [(1, 8), (3, 1), (5, 7), (11, 12), (7, 1004), (37, 24), (1000, 264), (17, 2056),
                (9, 8200), (2049, 512), (2, 131080)]


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
@pytest.mark.parametrize("rows,hidden", GEGLU_SHAPES)
def test_geglu_formats_shapes(dtype, rows, hidden):
    f = "f16" if dtype == np.float16 else "f32"
    x = synth.normal_with_outliers_bf16(3100 + rows + hidden, rows * 2 * hidden, 0.01, 50.0,
                                        fmt=f).reshape(rows, 2 * hidden)
    whole, out = guarded(rows * hidden, dtype)
    gpu_geglu(to_dev(x), rows, hidden, out, dtype)
    torch.cuda.synchronize()
    check_guard(whole, rows * hidden, dtype)
    assert_geglu_parity(out.cpu().numpy(), x, f"{rows}x{hidden}")


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_geglu_formats_unaligned_and_helper(dtype):
    f = "f16" if dtype == np.float16 else "f32"
    rows, hidden = 33, 1024
    x = synth.normal_bf16(52, 0, rows * 2 * hidden, fmt=f).reshape(rows, 2 * hidden)
    xb = to_dev(np.concatenate([np.zeros(1, dtype), x.ravel()]))
    whole, out = guarded(rows * hidden + 1, dtype)
    gpu_geglu(xb[1:], rows, hidden, out[1:], dtype)
    torch.cuda.synchronize()
    check_guard(whole, rows * hidden + 1, dtype)
    assert_geglu_parity(out[1:].cpu().numpy(), x, "unaligned")
    t = to_dev(x).reshape(3, 11, 2 * hidden)
    y = L.geglu(t)
    torch.cuda.synchronize()
    assert y.shape == (3, 11, hidden) and y.dtype == TORCH[dtype]
    assert_geglu_parity(y.cpu().numpy(), x, "helper")
    assert L.ltxk_geglu_dt(out.data_ptr(), xb.data_ptr(), 0, hidden, CODES[dtype],
                           stream()) == L.OK


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_geglu_formats_value_one_is_gelu(dtype):
    """value == 1: GEGLU gives GELU of the gate bit for bit (the same fp32
    value rounded once; |value| < 2 never takes the exact path)."""
    f = "f16" if dtype == np.float16 else "f32"
    rows, hidden = 64, 1024
    g = synth.normal_with_outliers_bf16(62, rows * hidden, 0.01, 50.0, fmt=f).reshape(rows, hidden)
    x = np.concatenate([np.ones((rows, hidden), dtype), g], axis=1)
    a = torch.empty(rows * hidden, dtype=TORCH[dtype], device="cuda")
    b = torch.empty_like(a)
    gpu_geglu(to_dev(x), rows, hidden, a, dtype)
    gpu_gelu(to_dev(g), rows * hidden, b, dtype)
    torch.cuda.synchronize()
    ua, ub = a.cpu().numpy().view(UINT[dtype]), b.cpu().numpy().view(UINT[dtype])
    assert np.array_equal(ua, ub)


@pytest.mark.parametrize("name", ["geglu_f16", "geglu_f32"])
def test_geglu_formats_workload_full_size(name):
    case = synth.WORKLOADS[name][0]
    dtype = synth.FORMATS[case.dtype]
    x = synth.make_x(case)
    n = case.rows * case.hidden
    whole, out = guarded(n, dtype)
    gpu_geglu(to_dev(x), case.rows, case.hidden, out, dtype)
    torch.cuda.synchronize()
    check_guard(whole, n, dtype)
    assert_geglu_parity(out.cpu().numpy(), x, case.name)
