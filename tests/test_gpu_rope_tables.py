"""GPU parity of the cos/sin tables computed on the device from token
positions (ltxk_rope_tables), and of the fused RMSNorm + RoPE fed with them.

Tables: every value within 4 * 2^-24 of the oracle's fp64 cos / sin (the
double-float angle reduction and sincospif give about 2 * 2^-24), on the
3-axis video grid, 1D text, a wrapped token range, and coordinates of 2^24
and beyond (the fp64 reduction path).  The fused form reads its tables as
inputs, so fed with the device tables it must stay within 1 bf16 ulp of the
oracle given the same fp32 tables.
"""
import numpy as np
import pytest
import torch

import oracle
import rope_element_dit_gb300 as L
import synth
from oracle.compare import compare_bf16

pytestmark = pytest.mark.gpu

BOUND = 4 * 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


CASES = [  # tokens, head_dim, grid, pairs
    (6144, 64, (8, 24, 32), (10, 11, 11)),            # the video workload's grid
    (4096, 128, (4096, 1, 1), (64, 0, 0)),            # 1D text
    (2 * 96 + 17, 64, (2, 6, 8), (10, 11, 11)),       # more tokens than positions: wraps
    (300, 512, (300, 1, 1), (256, 0, 0)),             # the largest head_dim
    (77, 6, (7, 11, 1), (1, 2, 0)),                   # odd sizes, an empty axis
]


@pytest.mark.parametrize("tokens,head_dim,grid,pairs", CASES)
def test_tables_match_the_oracle(tokens, head_dim, grid, pairs):
    cos, sin = L.rope_tables(head_dim, grid, pairs, tokens=tokens)
    torch.cuda.synchronize()
    c, s = oracle.rope_tables(tokens, head_dim, grid, pairs)
    assert cos.shape == (tokens, head_dim // 2) and cos.dtype == torch.float32
    assert np.abs(cos.cpu().numpy() - c).max() <= BOUND
    assert np.abs(sin.cpu().numpy() - s).max() <= BOUND


def test_tables_beyond_2p24_coordinates():
    """Coordinates of 2^24 and more take the fp64 reduction."""
    tokens = (1 << 24) + 2048
    cos, sin = L.rope_tables(2, (1 << 25, 1, 1), (1, 0, 0), tokens=tokens)
    torch.cuda.synchronize()
    tail = slice(tokens - 4096, tokens)                 # both sides of 2^24
    c, s = oracle.rope_tables(tokens, 2, (1 << 25, 1, 1), (1, 0, 0))
    assert np.abs(cos[tail].cpu().numpy() - c[tail]).max() <= BOUND
    assert np.abs(sin[tail].cpu().numpy() - s[tail]).max() <= BOUND


@pytest.mark.parametrize("mode", [L.ROPE_INTERLEAVED, L.ROPE_SPLIT_HALF])
def test_fused_form_on_device_tables(mode):
    heads, D, grid, pairs = 32, 64, (8, 24, 32), (10, 11, 11)
    S = grid[0] * grid[1] * grid[2]
    rows = 2 * S
    x = synth.normal_bf16(601, 0, rows * heads * D).reshape(rows, heads * D)
    w = synth.normal_bf16(601, 2, heads * D, 1.0, 0.1)
    cos, sin = L.rope_tables(D, grid, pairs)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    wd = torch.from_numpy(w.view(np.int16)).cuda().view(torch.bfloat16)
    y = L.rms_norm_rope(xd, wd, cos, sin, heads, D, mode, 1e-6, seq_len=S)
    torch.cuda.synchronize()
    ref = oracle.rms_norm_rope(x, w, cos.cpu().numpy(), sin.cpu().numpy(), heads, D, mode, 1e-6,
                               table_rows=S)
    r = compare_bf16(y.view(torch.int16).cpu().numpy().view(np.uint16), ref)
    assert r["ok"], r


def test_zero_tokens_and_stream():
    cos = torch.empty(0, 32, device="cuda")
    assert L.ltxk_rope_tables(cos.data_ptr() or 256, cos.data_ptr() or 512, 0, 64, 1, 1, 1,
                              32, 0, 0, 1e4, None) == L.OK
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c1, s1 = L.rope_tables(64, (8, 24, 32), (10, 11, 11))
    s.synchronize()
    c0, s0 = L.rope_tables(64, (8, 24, 32), (10, 11, 11))
    torch.cuda.synchronize()
    assert torch.equal(c0, c1) and torch.equal(s0, s1)
