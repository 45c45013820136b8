"""GPU parity of the tanh-approximated GELU and of GEGLU ("cuda-kernels"
skill page, "Kernel-Specific Guidelines / GEGLU vs GELU") against the fp64
oracle, element by element, at most 1 bf16 ulp (NaN matches NaN).

The kernel evaluates the sigmoid form in fp32 (relative error ~1e-5) and
rounds once, so a difference can only be a neighbouring value at a rounding
midpoint.  GELU is checked on EVERY bf16 input (all 65536 patterns: zeros,
subnormals, the far tail where e^{2z} leaves fp32, infinities, NaNs); GEGLU on
every gate value against values spread over 2^-126 .. 2^126.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import rope_element_dit_gb300 as L
import synth
from oracle.compare import compare_bf16

pytestmark = pytest.mark.gpu

THREADS = min(32, os.cpu_count() or 1)
CANARY = 0x7FC1
GUARD = 64
ALL_BITS = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU parity tests need a CUDA device"
    torch.cuda.set_device(0)
    assert torch.cuda.get_device_capability(0) == (10, 3)


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def to_host(t):
    return t.cpu().numpy().view(np.uint16)


def guarded(n):
    whole = torch.full((n + 2 * GUARD,), CANARY, dtype=torch.int16, device="cuda")
    return whole, whole[GUARD:GUARD + n]


def check_guard(whole, n):
    h = to_host(whole)
    assert np.all(h[:GUARD] == CANARY) and np.all(h[GUARD + n:] == CANARY), \
        "kernel wrote outside its output"


def stream():
    return torch.cuda.current_stream().cuda_stream


def assert_parity(got, ref, what, chunk=1 << 26):
    got, ref = got.reshape(-1), ref.reshape(-1)
    assert got.size == ref.size
    for s in range(0, got.size, chunk):
        r = compare_bf16(got[s:s + chunk], ref[s:s + chunk])
        assert r["ok"], f"{what}[{s}:]: {r}"


def gpu_gelu(x_dev, n, out):
    st = L.ltxk_gelu_tanh(out.data_ptr(), x_dev.data_ptr(), n, stream())
    assert st == L.OK, L.ltxk_status_string(st)


def gpu_geglu(x_dev, rows, hidden, out):
    st = L.ltxk_geglu(out.data_ptr(), x_dev.data_ptr(), rows, hidden, stream())
    assert st == L.OK, L.ltxk_status_string(st)


def wide_values(seed, n, lo=-126.0, hi=126.0):
    """bf16 values of random sign with log2-magnitude uniform in [lo, hi]."""
    e = synth.uniform_bf16(seed, 0, n, lo, hi)
    sign = synth.uniform_bf16(seed, 1, n, -1.0, 1.0)
    v = np.sign(synth.bf16_bits_to_f32(sign)) * np.exp2(synth.bf16_bits_to_f32(e))
    return synth.to_bf16_bits(v.astype(np.float32))


# -------------------------------------------------------------------- GELU --

@pytest.mark.parametrize("offset", [0, 1, 3])
def test_gelu_every_bf16_value(offset):
    """All 65536 inputs; offset 1 and 3 put the pointers off 16 bytes (element
    kernel), offset 0 takes the vector kernel."""
    n = ALL_BITS.size
    xb = to_dev(np.concatenate([np.zeros(offset, np.uint16), ALL_BITS]))
    whole, out = guarded(n + offset)
    gpu_gelu(xb[offset:], n, out[offset:])
    torch.cuda.synchronize()
    check_guard(whole, n + offset)
    assert_parity(to_host(out[offset:]), oracle.gelu_tanh(ALL_BITS), f"offset {offset}")


def test_gelu_workload_full_size():
    case = synth.GELU[0]
    x = synth.make_x(case)
    n = x.size
    whole, out = guarded(n)
    xd = to_dev(x)
    gpu_gelu(xd, n, out)
    torch.cuda.synchronize()
    check_guard(whole, n)
    assert_parity(to_host(out), oracle.gelu_tanh(x, threads=THREADS), case.name)


@pytest.mark.parametrize("n", [1, 7, 8, 9, 4095, 4096, 4097, 65543, 1000003])
def test_gelu_ragged_sizes(n):
    x = synth.normal_with_outliers_bf16(2000 + n, n, 0.01, 50.0)
    whole, out = guarded(n)
    xd = to_dev(x)
    gpu_gelu(xd, n, out)
    torch.cuda.synchronize()
    check_guard(whole, n)
    assert_parity(to_host(out), oracle.gelu_tanh(x), f"n={n}")


@pytest.mark.parametrize("n", [4096 * 3 + 5, 64])
def test_gelu_in_place(n):
    x = synth.uniform_bf16(31, 0, n, -12.0, 6.0)
    xd = to_dev(x)
    gpu_gelu(xd, n, xd)
    torch.cuda.synchronize()
    assert_parity(to_host(xd), oracle.gelu_tanh(x), "in place")


def test_gelu_zero_length_and_helper():
    xd = to_dev(np.zeros(8, np.uint16))
    assert L.ltxk_gelu_tanh(xd.data_ptr(), xd.data_ptr(), 0, stream()) == L.OK
    x = synth.normal_bf16(32, 0, 3 * 5 * 1000).reshape(3, 5, 1000)
    t = to_dev(x).view(torch.bfloat16).reshape(3, 5, 1000)
    y = L.gelu_tanh(t)
    torch.cuda.synchronize()
    assert y.shape == t.shape and y.dtype == torch.bfloat16
    assert_parity(y.view(torch.int16).cpu().numpy().view(np.uint16), oracle.gelu_tanh(x),
                  "helper")


# ------------------------------------------------------------------- GEGLU --

@pytest.mark.parametrize("rows,hidden", [(1, 65536), (256, 256)])
def test_geglu_every_gate_value(rows, hidden):
    """Every bf16 gate once, against values of magnitude 2^-126 .. 2^126."""
    v = wide_values(41, ALL_BITS.size).reshape(rows, hidden)
    g = ALL_BITS.reshape(rows, hidden)
    x = np.concatenate([v, g], axis=1)
    whole, out = guarded(rows * hidden)
    xd = to_dev(x)
    gpu_geglu(xd, rows, hidden, out)
    torch.cuda.synchronize()
    check_guard(whole, rows * hidden)
    assert_parity(to_host(out), oracle.geglu(x), f"{rows}x{hidden}")


def test_geglu_workload_full_size():
    case = synth.GEGLU[0]
    x = synth.make_x(case)
    n = case.rows * case.hidden
    whole, out = guarded(n)
    xd = to_dev(x)
    gpu_geglu(xd, case.rows, case.hidden, out)
    torch.cuda.synchronize()
    check_guard(whole, n)
    assert_parity(to_host(out), oracle.geglu(x, threads=THREADS), case.name)


GEGLU_SHAPES = [(1, 8), (3, 1), (5, 7), (37, 24), (1000, 264), (17, 2056), (9, 8200),
                (2049, 512), (3, 12288), (2, 131080)]


@pytest.mark.parametrize("rows,hidden", GEGLU_SHAPES)
def test_geglu_shapes(rows, hidden):
    x = synth.normal_with_outliers_bf16(3000 + rows + hidden, rows * 2 * hidden, 0.01,
                                        50.0).reshape(rows, 2 * hidden)
    whole, out = guarded(rows * hidden)
    xd = to_dev(x)
    gpu_geglu(xd, rows, hidden, out)
    torch.cuda.synchronize()
    check_guard(whole, rows * hidden)
    assert_parity(to_host(out), oracle.geglu(x), f"{rows}x{hidden}")


def test_geglu_unaligned_zero_rows_and_helper():
    rows, hidden = 33, 1024
    x = synth.normal_bf16(51, 0, rows * 2 * hidden).reshape(rows, 2 * hidden)
    xb = to_dev(np.concatenate([np.zeros(1, np.uint16), x.ravel()]))
    whole, out = guarded(rows * hidden + 1)
    gpu_geglu(xb[1:], rows, hidden, out[1:])
    torch.cuda.synchronize()
    check_guard(whole, rows * hidden + 1)
    ref = oracle.geglu(x)
    assert_parity(to_host(out[1:]), ref, "unaligned")
    assert L.ltxk_geglu(out.data_ptr(), xb.data_ptr(), 0, hidden, stream()) == L.OK
    t = to_dev(x).view(torch.bfloat16).reshape(3, 11, 2 * hidden)
    y = L.geglu(t)
    torch.cuda.synchronize()
    assert y.shape == (3, 11, hidden)
    assert_parity(y.view(torch.int16).cpu().numpy().view(np.uint16), ref, "helper")


def test_geglu_equals_value_times_gelu_when_value_is_one():
    """value == 1 everywhere: GEGLU's output is GELU of the gate, bit for bit
    (both kernels round the same fp32 product once)."""
    rows, hidden = 64, 1024
    g = synth.normal_with_outliers_bf16(61, rows * hidden, 0.01, 50.0).reshape(rows, hidden)
    one = np.full((rows, hidden), 0x3F80, np.uint16)
    xd = to_dev(np.concatenate([one, g], axis=1))
    gd = to_dev(g)
    a = torch.empty(rows * hidden, dtype=torch.int16, device="cuda")
    b = torch.empty_like(a)
    gpu_geglu(xd, rows, hidden, a)
    gpu_gelu(gd, rows * hidden, b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
