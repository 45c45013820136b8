"""The seeded input generator: reproducible, chunk-independent, and drawing
the distributions and table structure the workloads name."""
import numpy as np
import pytest

import synth


def test_splitmix64_reference_outputs():
    # SplitMix64 started from state 0: the first outputs of the published
    # generator (Steele, Lea & Flood 2014; same sequence as Vigna's
    # splitmix64.c with x = 0).
    z = synth.raw(np.uint64(0), 0, 3)
    assert [hex(int(v)) for v in z] == [
        "0xe220a8397b1dcdaf", "0x6e789e6aa1b965f4", "0x6c45d188009454f"]


def test_streams_reproducible_and_chunk_independent(monkeypatch):
    a = synth.normal_bf16(3, 0, 10_000)
    b = synth.normal_bf16(3, 0, 10_000)
    assert np.array_equal(a, b)
    monkeypatch.setattr(synth, "_CHUNK", 777)
    c = synth.normal_bf16(3, 0, 10_000, threads=3)
    assert np.array_equal(a, c)
    u1 = synth.uniform_bf16(3, 0, 5000, -4, 4)
    monkeypatch.setattr(synth, "_CHUNK", 1 << 22)
    assert np.array_equal(u1, synth.uniform_bf16(3, 0, 5000, -4, 4))


def test_streams_differ_by_seed_and_stream():
    assert not np.array_equal(synth.normal_bf16(1, 0, 64), synth.normal_bf16(2, 0, 64))
    assert not np.array_equal(synth.normal_bf16(1, 0, 64), synth.normal_bf16(1, 2, 64))


def test_distributions():
    f = synth.bf16_bits_to_f32(synth.normal_bf16(0, 0, 1 << 20)).astype(np.float64)
    assert abs(f.mean()) < 5e-3 and abs(f.std() - 1) < 5e-3
    w = synth.bf16_bits_to_f32(synth.normal_bf16(0, 2, 1 << 18, 1.0, 0.1))
    assert abs(w.mean() - 1) < 2e-3 and abs(w.std() - 0.1) < 2e-3
    u = synth.bf16_bits_to_f32(synth.uniform_bf16(7, 0, 1 << 20, -4, 4))
    assert u.min() >= -4 and u.max() <= 4 and abs(u.mean()) < 2e-2
    o = synth.bf16_bits_to_f32(synth.normal_with_outliers_bf16(1, 1 << 20, 0.01, 50.0))
    assert 0.006 < (np.abs(o) > 8).mean() < 0.01   # ~1% scaled, most land > 8


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    v = np.random.default_rng(0).standard_normal(1 << 16) * 1e3
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(synth.to_bf16_bits(v),
                          ref.view(torch.int16).numpy().view(np.uint16))


def test_rope_table_1d_structure():
    cos, sin = synth.rope_table_1d(4096, 128)
    assert cos.shape == (4096, 64) and cos.dtype == np.float32
    assert np.all(cos[0] == 1) and np.all(sin[0] == 0)        # position 0
    # pair 0 has frequency 1: angle = position
    s = np.arange(4096, dtype=np.float64)
    assert np.array_equal(cos[:, 0], np.cos(s).astype(np.float32))
    # frequencies fall with the pair index: first-row angles decrease
    ang = np.arctan2(sin[1].astype(np.float64), cos[1].astype(np.float64))
    assert np.all(np.diff(ang) < 0)
    np.testing.assert_allclose(cos.astype(np.float64) ** 2 + sin.astype(np.float64) ** 2,
                               1.0, atol=2e-7)


def test_rope_table_3axis_structure():
    cos, sin = synth.rope_table_3axis(8, 24, 32, 64)
    assert cos.shape == (6144, 32)
    assert np.all(cos[0] == 1) and np.all(sin[0] == 0)        # (0, 0, 0)
    # token (t, h, w) = (0, 0, 1): only the w-axis pairs (21..31) turn
    tok = 1
    assert np.all(sin[tok, :21] == 0) and np.all(sin[tok, 21:] != 0)
    # token (0, 1, 0) = 32: only the h-axis pairs (10..20) turn
    tok = 32
    assert np.all(sin[tok, :10] == 0) and np.all(sin[tok, 21:] == 0)
    assert np.all(sin[tok, 10:21] != 0)
    # token (1, 0, 0) = 768: only the t-axis pairs (0..9) turn; pair 0 by 1 rad
    tok = 768
    assert np.all(sin[tok, 10:] == 0)
    assert cos[tok, 0] == np.float32(np.cos(1.0))


def test_workloads_shapes():
    names = {c.name: c for cases in synth.WORKLOADS.values() for c in cases}
    assert names["rms_norm_4x4096x3072"].rows == 16384
    assert names["rms_norm_262143x2560"].rows == 262143
    r = names["rms_norm_rope_interleaved_2x4096x32x128"]
    assert r.heads * r.head_dim == r.hidden and r.rows == 2 * r.seq_len
    s = names["rms_norm_split_rope_1x6144x32x64"]
    assert s.heads * s.head_dim == s.hidden and s.rows == s.seq_len
    assert [c.seed for c in synth.SWEEP] == [1, 2, 3, 4]
    assert [c.seed for c in synth.STRESS] == [7, 8, 9]


def test_algorithmic_bytes():
    c = synth.SWEEP[-1]
    assert synth.algorithmic_bytes(c) == 4 * 16384 * 3072 + 2 * 3072
    r = synth.ROPE_INTERLEAVED[0]
    assert synth.algorithmic_bytes(r) == 4 * 8192 * 4096 + 2 * 4096 + 8 * 4096 * 64
    assert synth.algorithmic_bytes(r, per_row_tables=True) == (
        4 * 8192 * 4096 + 2 * 4096 + 8 * 8192 * 64)
