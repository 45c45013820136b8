"""GPU parity at the sizes where 32-bit element indexing would break: calls
of more than 2^31 elements (4.3 GB of bf16 in, 4.3 GB out), and rows of the
largest hidden size the boundary accepts (LTXK_MAX_HIDDEN = 2^30 elements).

Rows are independent, so a call over a tiled input (row r is row r mod B of
a seeded block) is checked row by row on a sample: the first rows, the rows
around element 2^31, the last rows and seeded random rows, each against the
oracle of its block row.  The maximum-hidden rows are checked whole.
"""
import numpy as np
import pytest
import torch

import oracle
import rope_element_dit_gb300 as L
import synth
from oracle.compare import compare_bf16, compare_bf16_bounded

pytestmark = pytest.mark.gpu

THREADS = 16
BLOCK = 4096          # rows of the seeded block the big inputs tile


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU parity tests need a CUDA device"
    torch.cuda.set_device(0)
    assert torch.cuda.get_device_capability(0) == (10, 3)
    yield
    torch.cuda.empty_cache()


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def tiled(block_bits, rows):
    """[rows, hidden] on the device, row r = block row r mod len(block)."""
    b = bf16_dev(block_bits)
    reps = -(-rows // b.shape[0])
    return b.repeat(reps, 1)[:rows].contiguous()


def sample_rows(rows, hidden, seed):
    """First, last, around element 2^31, and 61 seeded random rows."""
    edge = (1 << 31) // hidden
    fixed = [0, 1, 2, edge - 2, edge - 1, edge, edge + 1, edge + 2, rows - 2, rows - 1]
    rng = np.random.default_rng(seed)
    picked = np.concatenate([fixed, rng.integers(0, rows, 61)])
    return np.unique(picked[(picked >= 0) & (picked < rows)])


def gathered(y, idx):
    return host_bits(y.index_select(0, torch.from_numpy(idx).cuda()))


def test_rms_norm_beyond_2p31_elements():
    rows, hidden = (1 << 20) + 3, 2048                    # 2^31 + 6144 elements
    assert rows * hidden > 1 << 31
    block = synth.normal_with_outliers_bf16(301, BLOCK * hidden, 0.01, 50.0).reshape(BLOCK, hidden)
    w = synth.normal_bf16(301, 2, hidden, 1.0, 0.1)
    x = tiled(block, rows)
    y = L.rms_norm(x, bf16_dev(w), 1e-6)
    torch.cuda.synchronize()
    idx = sample_rows(rows, hidden, 302)
    ref = oracle.rms_norm(block[idx % BLOCK], w, 1e-6, threads=THREADS)
    r = compare_bf16(gathered(y, idx), ref)
    assert r["ok"], r
    del x, y


@pytest.mark.parametrize("mode", [L.ROPE_INTERLEAVED, L.ROPE_SPLIT_HALF])
def test_rms_norm_rope_beyond_2p31_elements(mode):
    heads, D, S = 32, 128, 4096
    hidden = heads * D
    rows = (1 << 19) + 5                                  # 2^31 + 20480 elements
    block = synth.normal_bf16(303, 0, BLOCK * hidden).reshape(BLOCK, hidden)
    w = synth.normal_bf16(303, 2, hidden, 1.0, 0.1)
    cos, sin = synth.rope_table_1d(S, D)
    x = tiled(block, rows)
    y = L.rms_norm_rope(x, bf16_dev(w), torch.from_numpy(cos).cuda(),
                        torch.from_numpy(sin).cuda(), heads, D, mode, 1e-6, seq_len=S)
    torch.cuda.synchronize()
    idx = sample_rows(rows, hidden, 304)
    # row r uses table row r mod S; BLOCK == S, so the block row and its
    # position coincide for every sampled row
    ref = oracle.rms_norm_rope(block[idx % BLOCK], w, cos[idx % S], sin[idx % S], heads, D,
                               mode, 1e-6, threads=THREADS)
    r = compare_bf16(gathered(y, idx), ref)
    assert r["ok"], r
    del x, y


def test_rope_positions_beyond_2p31_elements():
    heads, D, T = 32, 128, 4096
    hidden = heads * D
    rows = (1 << 19) + 5
    block = synth.normal_bf16(305, 0, BLOCK * hidden).reshape(BLOCK, hidden)
    x = tiled(block, rows)
    y = L.rope(x, heads, D, L.ROPE_INTERLEAVED, (T, 1, 1), (D // 2, 0, 0))
    torch.cuda.synchronize()
    idx = sample_rows(rows, hidden, 306)
    # token s = r mod T; BLOCK == T, so row r of the call is row r mod T of
    # the block, and the oracle over the whole block numbers its rows (and
    # positions) 0 .. T-1
    _, ye_block = oracle.rope(block, heads, D, 0, (T, 1, 1), (D // 2, 0, 0), exact=True,
                              threads=THREADS)
    ye = ye_block[idx % BLOCK]
    xa = np.abs(oracle.widen_bf16(block[idx % BLOCK])).reshape(len(idx), heads, D // 2, 2)
    m = np.repeat(xa.sum(axis=-1), 2, axis=-1).reshape(len(idx), hidden)
    r = compare_bf16_bounded(gathered(y, idx), ye, 8 * 2.0 ** -24 * m)
    assert r["ok"], r
    del x, y


def test_gelu_beyond_2p31_elements():
    n = (1 << 31) + (1 << 19) + 9
    chunk = synth.normal_with_outliers_bf16(307, 1 << 20, 0.01, 50.0)
    x = bf16_dev(chunk).repeat(-(-n // chunk.size))[:n].contiguous()
    y = L.gelu_tanh(x)
    torch.cuda.synchronize()
    ref = oracle.gelu_tanh(chunk)
    # 2^20-element windows: the start, across element 2^31, and the end (with
    # the one-element tail the element kernel takes)
    for start in (0, (1 << 31) - (1 << 19), n - (1 << 20)):
        got = host_bits(y[start:start + (1 << 20)])
        want = np.roll(ref, -(start % chunk.size))
        r = compare_bf16(got, want)
        assert r["ok"], (start, r)
    del x, y


def test_rms_norm_largest_hidden():
    """Two rows of LTXK_MAX_HIDDEN = 2^30 elements (2 GiB each): the
    element-wise kernel, 64-bit offsets inside a row, checked whole."""
    hidden, rows = 1 << 30, 2
    p0 = synth.normal_bf16(309, 0, 1 << 20)
    p1 = synth.uniform_bf16(309, 1, 1 << 20, -4.0, 4.0)
    xh = np.stack([np.tile(p0, hidden // p0.size), np.tile(p1, hidden // p1.size)])
    x = bf16_dev(xh)
    y = L.rms_norm(x, None, 1e-6)
    torch.cuda.synchronize()
    yh = host_bits(y)
    del x, y
    torch.cuda.empty_cache()
    ref = oracle.rms_norm(xh, None, 1e-6, threads=2)
    for r0 in range(rows):
        for s in range(0, hidden, 1 << 27):
            r = compare_bf16(yh[r0, s:s + (1 << 27)], ref[r0, s:s + (1 << 27)])
            assert r["ok"], (r0, s, r)
