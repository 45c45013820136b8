"""A missing weight and a weight of ones give the same bits.

`w == NULL` means a weight of ones (the pages' `elementwise_affine=False`
norms, "Diffusers Critical Pitfalls").  The row kernels compile their
epilogue twice, with and without a weight, and skip every weight load and
product when there is none; since x * 1 = x exactly, both forms must agree
bit for bit, in every row operation, element format and kernel family
(vector, element-wise), for ragged and full rows.  The oracle comparisons
of the same calls are in the parity tests; this pins the specialisation
itself.
"""
import numpy as np
import pytest
import torch

import rope_element_dit_gb300 as L
import synth

pytestmark = pytest.mark.gpu

FMTS = {"bf16": (torch.bfloat16, L.DTYPE_BF16), "f16": (torch.float16, L.DTYPE_F16),
        "f32": (torch.float32, L.DTYPE_F32)}


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


def s():
    return torch.cuda.current_stream().cuda_stream


def rows_of(fmt, seed, rows, hidden):
    a = synth.normal_with_outliers_bf16(seed, rows * hidden, 0.01, 50.0, fmt=fmt)
    if fmt == "bf16":
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def ones(fmt, n):
    return torch.ones(n, dtype=FMTS[fmt][0], device="cuda")


def same_bits(a, b):
    ia = a.view(torch.int16 if a.element_size() == 2 else torch.int32)
    ib = b.view(torch.int16 if b.element_size() == 2 else torch.int32)
    return bool(torch.equal(ia, ib))


# (rows, hidden): vector kernels with one, two and four warps per row, a
# ragged last vector slot, and the element-wise kernel (hidden % 8 != 0)
SHAPES = [(300, 2048), (37, 3072), (1000, 4096), (9, 264), (5, 1000), (7, 6)]


@pytest.mark.parametrize("fmt", list(FMTS))
@pytest.mark.parametrize("rows,hidden", SHAPES)
def test_rms_norm_and_adaln_and_add_norm(fmt, rows, hidden):
    dt = FMTS[fmt][1]
    x = rows_of(fmt, 7100 + hidden, rows, hidden)
    one = ones(fmt, hidden)
    y0, y1 = torch.empty_like(x), torch.empty_like(x)
    assert L.ltxk_rms_norm_dt(y0.data_ptr(), x.data_ptr(), None, rows, hidden, 1e-6, dt,
                              s()) == L.OK
    assert L.ltxk_rms_norm_dt(y1.data_ptr(), x.data_ptr(), one.data_ptr(), rows, hidden, 1e-6,
                              dt, s()) == L.OK
    torch.cuda.synchronize()
    assert same_bits(y0, y1), "rms_norm"
    rpc = max(1, rows // 3)
    ncond = -(-rows // rpc)
    sc = rows_of(fmt, 7200 + hidden, ncond, hidden) * 0.01
    sh = rows_of(fmt, 7300 + hidden, ncond, hidden) * 0.01
    assert L.ltxk_rms_norm_adaln_dt(y0.data_ptr(), x.data_ptr(), None, sc.data_ptr(),
                                    sh.data_ptr(), rows, hidden, rpc, 1e-6, dt, s()) == L.OK
    assert L.ltxk_rms_norm_adaln_dt(y1.data_ptr(), x.data_ptr(), one.data_ptr(), sc.data_ptr(),
                                    sh.data_ptr(), rows, hidden, rpc, 1e-6, dt, s()) == L.OK
    torch.cuda.synchronize()
    assert same_bits(y0, y1), "adaln"
    res = rows_of(fmt, 7400 + hidden, rows, hidden)
    h0, h1 = torch.empty_like(x), torch.empty_like(x)
    assert L.ltxk_add_rms_norm_dt(y0.data_ptr(), h0.data_ptr(), x.data_ptr(), res.data_ptr(),
                                  None, rows, hidden, 1e-6, dt, s()) == L.OK
    assert L.ltxk_add_rms_norm_dt(y1.data_ptr(), h1.data_ptr(), x.data_ptr(), res.data_ptr(),
                                  one.data_ptr(), rows, hidden, 1e-6, dt, s()) == L.OK
    torch.cuda.synchronize()
    assert same_bits(h0, h1) and same_bits(y0, y1), "add_rms_norm"


# (rows, heads, head_dim, seq_len): vector rotation kernels (interleaved
# head_dim % 8, split-half % 16) and the element-wise one (head_dim 6)
ROPE = [(128, 32, 128, 64), (300, 32, 64, 100), (33, 4, 16, 11), (17, 5, 6, 17)]


@pytest.mark.parametrize("fmt", list(FMTS))
@pytest.mark.parametrize("rows,heads,D,seq_len", ROPE)
@pytest.mark.parametrize("mode", [L.ROPE_INTERLEAVED, L.ROPE_SPLIT_HALF])
def test_rms_norm_rope(fmt, rows, heads, D, seq_len, mode):
    dt = FMTS[fmt][1]
    H = heads * D
    x = rows_of(fmt, 7500 + D, rows, H)
    one = ones(fmt, H)
    c, sn = synth.rope_table_1d(seq_len, D)
    c, sn = torch.from_numpy(c).cuda(), torch.from_numpy(sn).cuda()
    y0, y1 = torch.empty_like(x), torch.empty_like(x)
    for y, w in ((y0, None), (y1, one.data_ptr())):
        assert L.ltxk_rms_norm_rope_dt(y.data_ptr(), x.data_ptr(), w, c.data_ptr(), sn.data_ptr(),
                                       rows, heads, D, mode, 1e-6, seq_len, dt, s()) == L.OK
    torch.cuda.synchronize()
    assert same_bits(y0, y1)
