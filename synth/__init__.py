"""Seeded synthetic inputs for bf16 RMSNorm and fused RMSNorm+RoPE.

This module is shared by the tests, the benchmark and the smoke check.  It
holds none of the operation's arithmetic: it only draws random activations and
weights, rounds them to bfloat16, and builds the binary32 cos/sin tables that
the fused operation takes as inputs.  It imports neither the CUDA binding nor
the oracle.

Random numbers
--------------
The pages name no generator, so "seed k" means the following counter-based
stream, defined here once:

* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): the i-th output (i = 0, 1, ...) of the stream
  with key K is mix(K + (i + 1) * 0x9E3779B97F4A7C15), where
  mix(z): z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
          z *= 0x94D049BB133111EB; z ^= z >> 31   (all mod 2^64).
* Each tensor has its own stream: K = mix(seed * 2^8 + stream_id), with
  stream ids X=0 (activations), OUTLIER=1 (outlier selection), WEIGHT=2.
  Because outputs are indexed, any chunk of a tensor can be drawn on its own.
* Uniform on [0, 1): (z >> 11) * 2^-53.  Uniform on (0, 1]: ((z >> 11) + 1) *
  2^-53.
* N(0, 1): Box-Muller, cosine branch only: element k uses outputs 2k and 2k+1,
  n_k = sqrt(-2 ln u1) * cos(2 pi u0), with u1 on (0, 1] and u0 on [0, 1).
* Values are drawn in binary64, cast to binary32 (round to nearest even) and
  then to bfloat16 (round to nearest even on the binary32 bits).

The integer stream is bit-exact on every host.  The normal draws go through
numpy's log/cos/sqrt, which may differ in the last bit of a binary64 value
between platforms; that very rarely changes a bfloat16 input, and parity never
depends on it because the oracle and the CUDA path read the same arrays.

bfloat16 tensors are returned as numpy.uint16 arrays of bit patterns.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)

STREAM_X = 0
STREAM_OUTLIER = 1
STREAM_WEIGHT = 2

INTERLEAVED = 0
SPLIT_HALF = 1

_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * M1
    z = z ^ (z >> np.uint64(27))
    z = z * M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        return _mix(np.array([(seed << 8) + stream], dtype=np.uint64))[0]


def raw(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the SplitMix64 stream with ``key``."""
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + i * GAMMA)


def _unit_open_right(z):   # [0, 1)
    return (z >> np.uint64(11)).astype(np.float64) * 2.0 ** -53


def _unit_open_left(z):    # (0, 1]
    return ((z >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * 2.0 ** -53


def to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """binary64 -> binary32 (RNE) -> bfloat16 bits (RNE on the binary32 bits)."""
    f = np.ascontiguousarray(v, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact binary32 values of bfloat16 bit patterns (for statistics)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# Element formats of generated arrays: bf16 as uint16 bit patterns, the other
# two as numpy floats (binary64 -> format, round to nearest even).
FORMATS = {"bf16": np.uint16, "f16": np.float16, "f32": np.float32}


def to_format(v: np.ndarray, fmt: str) -> np.ndarray:
    if fmt == "bf16":
        return to_bf16_bits(v)
    return np.asarray(v, dtype=np.float64).astype(FORMATS[fmt])


def _chunked(n: int, fn, threads: int | None, fmt: str = "bf16") -> np.ndarray:
    out = np.empty(n, dtype=FORMATS[fmt])
    starts = list(range(0, n, _CHUNK))
    if len(starts) <= 1:
        if n:
            out[:] = fn(0, n)
        return out
    threads = threads or min(32, os.cpu_count() or 1)

    def work(s):
        e = min(n, s + _CHUNK)
        out[s:e] = fn(s, e - s)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(work, starts))
    return out


def normal_bf16(seed: int, stream: int, n: int, mean: float = 0.0,
                std: float = 1.0, threads: int | None = None, fmt: str = "bf16",
                start: int = 0) -> np.ndarray:
    """n draws of N(mean, std^2), rounded to bfloat16 (bit patterns), or to
    float16 / float32 with ``fmt``: elements start .. start+n-1 of the
    stream (the stream is counter-based, so any slice is generated alone)."""
    key = stream_key(seed, stream)

    def fn(s, c):
        z = raw(key, 2 * (start + s), 2 * c)
        u0 = _unit_open_right(z[0::2])
        u1 = _unit_open_left(z[1::2])
        g = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u0)
        return to_format(mean + std * g, fmt)

    return _chunked(n, fn, threads, fmt)


def uniform_bf16(seed: int, stream: int, n: int, lo: float, hi: float,
                 threads: int | None = None, fmt: str = "bf16", start: int = 0) -> np.ndarray:
    """n draws of U[lo, hi), rounded to bfloat16 (bit patterns), or to
    float16 / float32 with ``fmt``: elements start .. start+n-1 of the stream."""
    key = stream_key(seed, stream)

    def fn(s, c):
        u = _unit_open_right(raw(key, start + s, c))
        return to_format(lo + (hi - lo) * u, fmt)

    return _chunked(n, fn, threads, fmt)


def normal_with_outliers_bf16(seed: int, n: int, frac: float, scale: float,
                              threads: int | None = None, fmt: str = "bf16",
                              start: int = 0) -> np.ndarray:
    """N(0,1) draws where each element, independently with probability
    ``frac`` (its own uniform from the OUTLIER stream), is multiplied by
    ``scale`` before the rounding to bfloat16 (or ``fmt``); elements
    start .. start+n-1."""
    kx = stream_key(seed, STREAM_X)
    ko = stream_key(seed, STREAM_OUTLIER)

    def fn(s, c):
        z = raw(kx, 2 * (start + s), 2 * c)
        g = (np.sqrt(-2.0 * np.log(_unit_open_left(z[1::2])))
             * np.cos(2.0 * math.pi * _unit_open_right(z[0::2])))
        sel = _unit_open_right(raw(ko, start + s, c)) < frac
        g = np.where(sel, g * scale, g)
        return to_format(g, fmt)

    return _chunked(n, fn, threads, fmt)


# ---- rotary tables (inputs of the fused operation) -------------------------

def rope_table_1d(seq_len: int, head_dim: int, theta: float = 10000.0):
    """cos/sin [seq_len, head_dim/2] for 1-D positions 0..seq_len-1.

    Pair p uses frequency theta^(-2p/head_dim); angle = position * frequency.
    Computed in binary64, stored as binary32.
    """
    P = head_dim // 2
    inv = theta ** (-2.0 * np.arange(P, dtype=np.float64) / head_dim)
    ang = np.arange(seq_len, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def rope_table_3axis(t: int, h: int, w: int, head_dim: int,
                     pairs_per_axis=(10, 11, 11), theta: float = 10000.0):
    """cos/sin [t*h*w, head_dim/2] for video tokens on a (t, h, w) grid.

    Token s = (ti*h + hi)*w + wi.  The head_dim/2 pairs are split into
    consecutive groups, one per axis (t, then h, then w); inside an axis with
    n pairs, pair k uses frequency theta^(-k/n) and angle = coordinate *
    frequency.  Computed in binary64, stored as binary32.
    """
    P = head_dim // 2
    if sum(pairs_per_axis) != P:
        raise ValueError("pairs_per_axis must add up to head_dim/2")
    ti, hi, wi = np.meshgrid(np.arange(t), np.arange(h), np.arange(w),
                             indexing="ij")
    coords = [a.reshape(-1).astype(np.float64) for a in (ti, hi, wi)]
    cols = []
    for coord, n in zip(coords, pairs_per_axis):
        inv = theta ** (-np.arange(n, dtype=np.float64) / n)
        cols.append(coord[:, None] * inv[None, :])
    ang = np.concatenate(cols, axis=1)
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


# ---- the workloads ---------------------------------------------------------

@dataclass
class Case:
    """One seeded input set.  ``mode`` is None for plain RMSNorm."""
    name: str
    rows: int
    hidden: int
    seed: int
    x_dist: str                    # "normal", "normal_outliers", "uniform4"
    eps: float
    mode: int | None = None
    heads: int = 0
    head_dim: int = 0
    seq_len: int = 0               # positions per batch item (table rows)
    table: str = ""                # "1d" or "3axis"
    meta: dict = field(default_factory=dict)
    op: str = ""                   # "adaln", "add_norm", "gelu", "geglu", "rope_pos"
    weight: bool = True            # False: no weight (ones)
    rows_per_cond: int = 0         # AdaLN: rows sharing one conditioning row
    dtype: str = "bf16"            # element format of x, w, scale, shift, res

    @property
    def elements(self) -> int:
        return self.rows * self.hidden

    @property
    def in_width(self) -> int:
        """Elements per input row: 2 * hidden for GEGLU (value, gate)."""
        return 2 * self.hidden if self.op == "geglu" else self.hidden

    @property
    def kind(self) -> str:
        if self.op:
            return self.op
        return "norm" if self.mode is None else "rope"

    @property
    def n_cond(self) -> int:
        return -(-self.rows // self.rows_per_cond) if self.rows_per_cond else 0


def _norm(name, b, s, h, seed, dist, eps):
    return Case(name=name, rows=b * s, hidden=h, seed=seed, x_dist=dist,
                eps=eps, meta={"shape": [b, s, h]})


# RMSNorm on [1x1024x2048], N(0,1) activations, seed 0.
SMALL = [_norm("rms_norm_1x1024x2048", 1, 1024, 2048, 0, "normal", 1e-6)]

# RMSNorm shape sweep with 1 % x50 outliers, seeds 1..4 in listed order.
SWEEP = [
    _norm("rms_norm_2x1024x2048", 2, 1024, 2048, 1, "normal_outliers", 1e-6),
    _norm("rms_norm_4x1024x2048", 4, 1024, 2048, 2, "normal_outliers", 1e-6),
    _norm("rms_norm_2x4096x3072", 2, 4096, 3072, 3, "normal_outliers", 1e-6),
    _norm("rms_norm_4x4096x3072", 4, 4096, 3072, 4, "normal_outliers", 1e-6),
]

# Fused RMSNorm + interleaved RoPE, [2, 4096, 32 heads x 128], 1-D positions.
ROPE_INTERLEAVED = [Case(
    name="rms_norm_rope_interleaved_2x4096x32x128", rows=2 * 4096,
    hidden=4096, seed=5, x_dist="normal", eps=1e-6, mode=INTERLEAVED,
    heads=32, head_dim=128, seq_len=4096, table="1d",
    meta={"shape": [2, 4096, 4096], "theta": 10000.0})]

# Fused RMSNorm + split-half RoPE, [1, 6144 video tokens, 32 heads x 64],
# positions on an 8 x 24 x 32 grid, pairs 10/11/11 per axis.
ROPE_SPLIT = [Case(
    name="rms_norm_split_rope_1x6144x32x64", rows=6144, hidden=2048, seed=6,
    x_dist="normal", eps=1e-6, mode=SPLIT_HALF, heads=32, head_dim=64,
    seq_len=6144, table="3axis",
    meta={"shape": [1, 6144, 2048], "grid": [8, 24, 32],
          "pairs_per_axis": [10, 11, 11], "theta": 10000.0})]

# Bandwidth stress and ragged tails, U(-4,4), eps 1e-5, seeds 7..9.
STRESS = [
    _norm("rms_norm_4x16384x4096", 4, 16384, 4096, 7, "uniform4", 1e-5),
    _norm("rms_norm_262143x2560", 1, 262143, 2560, 8, "uniform4", 1e-5),
    _norm("rms_norm_65536x5120", 1, 65536, 5120, 9, "uniform4", 1e-5),
]

# AdaLN-modulated RMSNorm, x [2, 6144, 2048] with no weight (the pages'
# weightless LTX-Video block norm); scale, shift [2, 2048] ~ N(0, 0.5).
ADALN = [Case(
    name="rms_norm_adaln_2x6144x2048", rows=2 * 6144, hidden=2048, seed=10,
    x_dist="normal", eps=1e-6, op="adaln", weight=False, rows_per_cond=6144,
    meta={"shape": [2, 6144, 2048], "cond": [2, 2048], "scale_std": 0.5,
          "shift_std": 0.5})]

# Fused residual add + RMSNorm on the largest sweep shape [4, 4096, 3072]:
# x, residual ~ N(0, 1), weight ~ N(1, 0.1).
ADD_NORM = [Case(
    name="add_rms_norm_4x4096x3072", rows=4 * 4096, hidden=3072, seed=11,
    x_dist="normal", eps=1e-6, op="add_norm", meta={"shape": [4, 4096, 3072]})]

# Tanh-approximated GELU and GEGLU of an LTX-Video-sized feed-forward block:
# 2 x 6144 tokens, inner width 4 x 2048 = 8192; pre-activations N(0, 1) with
# 1 % x50 outliers, which also reach the far negative tail.
GELU = [Case(
    name="gelu_tanh_2x6144x8192", rows=2 * 6144, hidden=8192, seed=12,
    x_dist="normal_outliers", eps=0.0, op="gelu", weight=False,
    meta={"shape": [2, 6144, 8192]})]

GEGLU = [Case(
    name="geglu_2x6144x16384", rows=2 * 6144, hidden=8192, seed=13,
    x_dist="normal_outliers", eps=0.0, op="geglu", weight=False,
    meta={"shape": [2, 6144, 16384], "out_shape": [2, 6144, 8192]})]

# GELU and GEGLU in the pages' other two precision modes, on the same
# feed-forward shapes and recipe.
GELU_F16 = [Case(
    name="gelu_tanh_f16_2x6144x8192", rows=2 * 6144, hidden=8192, seed=18,
    x_dist="normal_outliers", eps=0.0, op="gelu", weight=False, dtype="f16",
    meta={"shape": [2, 6144, 8192]})]
GELU_F32 = [Case(
    name="gelu_tanh_f32_2x6144x8192", rows=2 * 6144, hidden=8192, seed=19,
    x_dist="normal_outliers", eps=0.0, op="gelu", weight=False, dtype="f32",
    meta={"shape": [2, 6144, 8192]})]
GEGLU_F16 = [Case(
    name="geglu_f16_2x6144x16384", rows=2 * 6144, hidden=8192, seed=20,
    x_dist="normal_outliers", eps=0.0, op="geglu", weight=False, dtype="f16",
    meta={"shape": [2, 6144, 16384], "out_shape": [2, 6144, 8192]})]
GEGLU_F32 = [Case(
    name="geglu_f32_2x6144x16384", rows=2 * 6144, hidden=8192, seed=21,
    x_dist="normal_outliers", eps=0.0, op="geglu", weight=False, dtype="f32",
    meta={"shape": [2, 6144, 16384], "out_shape": [2, 6144, 8192]})]

# The pages' other two precision modes on the largest sweep shape
# [4, 4096, 3072]: RMSNorm in float16 and in float32, N(0,1) with 1% x50
# outliers (the sweep's recipe), w ~ N(1, 0.1).
F16 = [Case(name="rms_norm_f16_4x4096x3072", rows=4 * 4096, hidden=3072, seed=14,
            x_dist="normal_outliers", eps=1e-6, dtype="f16", meta={"shape": [4, 4096, 3072]})]
F32 = [Case(name="rms_norm_f32_4x4096x3072", rows=4 * 4096, hidden=3072, seed=15,
            x_dist="normal_outliers", eps=1e-6, dtype="f32", meta={"shape": [4, 4096, 3072]})]

# Standalone RoPE with angles computed on the device from token positions,
# on the fused configs' shapes: 1D text [2, 4096, 32 x 128] interleaved and
# 3D video [1, 8x24x32, 32 x 64] split-half, theta 1e4, N(0,1), no weight.
ROPE_POS_TEXT = [Case(
    name="rope_pos_text_2x4096x32x128", rows=2 * 4096, hidden=4096, seed=16,
    x_dist="normal", eps=0.0, mode=INTERLEAVED, heads=32, head_dim=128, op="rope_pos",
    weight=False, meta={"shape": [2, 4096, 32, 128], "grid": [4096, 1, 1],
                        "pairs": [64, 0, 0], "theta": 10000.0})]
ROPE_POS_VIDEO = [Case(
    name="rope_pos_video_1x6144x32x64", rows=6144, hidden=2048, seed=17,
    x_dist="normal", eps=0.0, mode=SPLIT_HALF, heads=32, head_dim=64, op="rope_pos",
    weight=False, meta={"shape": [1, 6144, 32, 64], "grid": [8, 24, 32],
                        "pairs": [10, 11, 11], "theta": 10000.0})]

# The five configurations in one step: the bandwidth stress shapes (the
# largest problems) with the small case, the sweep and both fused forms.
FIVE_CONFIGS = SMALL + SWEEP + ROPE_INTERLEAVED + ROPE_SPLIT + STRESS

WORKLOADS = {
    "five_configs": FIVE_CONFIGS,
    "small": SMALL,
    "sweep": SWEEP,
    "rope_interleaved": ROPE_INTERLEAVED,
    "rope_split": ROPE_SPLIT,
    "stress": STRESS,
    "adaln": ADALN,
    "add_norm": ADD_NORM,
    "gelu": GELU,
    "geglu": GEGLU,
    "gelu_f16": GELU_F16,
    "gelu_f32": GELU_F32,
    "geglu_f16": GEGLU_F16,
    "geglu_f32": GEGLU_F32,
    "f16": F16,
    "f32": F32,
    "rope_pos_text": ROPE_POS_TEXT,
    "rope_pos_video": ROPE_POS_VIDEO,
}

STREAM_SCALE = 3
STREAM_SHIFT = 4
STREAM_RESIDUAL = 5


def make_x(case: Case, threads: int | None = None) -> np.ndarray:
    """x [rows, in_width]; for a shard (``shard_case``) the rows
    row_start .. row_start+rows-1 of the whole batch."""
    n = case.rows * case.in_width
    f = case.dtype
    o = case.meta.get("row_start", 0) * case.in_width
    if case.x_dist == "normal":
        x = normal_bf16(case.seed, STREAM_X, n, threads=threads, fmt=f, start=o)
    elif case.x_dist == "normal_outliers":
        x = normal_with_outliers_bf16(case.seed, n, 0.01, 50.0, threads=threads, fmt=f, start=o)
    elif case.x_dist == "uniform4":
        x = uniform_bf16(case.seed, STREAM_X, n, -4.0, 4.0, threads=threads, fmt=f, start=o)
    else:
        raise ValueError(case.x_dist)
    return x.reshape(case.rows, case.in_width)


def make_w(case: Case) -> np.ndarray:
    """Weight ~ N(1, 0.1), in the case's format."""
    return normal_bf16(case.seed, STREAM_WEIGHT, case.hidden, 1.0, 0.1, fmt=case.dtype)


def make_tables(case: Case):
    if case.mode is None or case.kind == "rope_pos":
        return None, None
    if case.table == "1d":
        return rope_table_1d(case.seq_len, case.head_dim,
                             case.meta.get("theta", 10000.0))
    if case.table == "3axis":
        t, h, w = case.meta["grid"]
        return rope_table_3axis(t, h, w, case.head_dim,
                                tuple(case.meta["pairs_per_axis"]),
                                case.meta.get("theta", 10000.0))
    raise ValueError(case.table)


def make_cond(case: Case):
    """AdaLN scale and shift, [n_cond, hidden] in the case's format (for a
    shard: the conditioning rows of its batch items)."""
    if case.kind != "adaln":
        return None, None
    n = case.n_cond * case.hidden
    o = case.meta.get("row_start", 0) // case.rows_per_cond * case.hidden
    sc = normal_bf16(case.seed, STREAM_SCALE, n, 0.0, case.meta.get("scale_std", 0.5),
                     fmt=case.dtype, start=o)
    sh = normal_bf16(case.seed, STREAM_SHIFT, n, 0.0, case.meta.get("shift_std", 0.5),
                     fmt=case.dtype, start=o)
    return sc.reshape(case.n_cond, case.hidden), sh.reshape(case.n_cond, case.hidden)


def make_inputs(case: Case, threads: int | None = None) -> dict:
    cos, sin = make_tables(case)
    scale, shift = make_cond(case)
    res = None
    if case.kind == "add_norm":
        res = normal_bf16(case.seed, STREAM_RESIDUAL, case.elements, threads=threads,
                          fmt=case.dtype, start=case.meta.get("row_start", 0) * case.hidden
                          ).reshape(case.rows, case.hidden)
    return {"x": make_x(case, threads), "w": make_w(case) if case.weight else None,
            "cos": cos, "sin": sin, "scale": scale, "shift": shift, "res": res}


def shard_rows(rows: int, world: int, rank: int):
    """Rows [r0, r1) of a batch that rank ``rank`` of ``world`` takes: rows
    are independent, so a contiguous split needs no exchange."""
    base, extra = divmod(rows, world)
    r0 = rank * base + min(rank, extra)
    return r0, r0 + base + (1 if rank < extra else 0)


def shard_case(case: Case, world: int, rank: int) -> Case:
    """Rank ``rank``'s part of a batch of ``world`` x the case's rows (the
    case as one GPU's share of a batch that grows with the GPU count).  The
    shard's rows are rows [r0, r1) of that batch, generated from the same
    counter-based streams; the weight and the tables are the case's own.
    A shard starts at a whole sequence (tables), a whole position grid
    (positions) and a whole batch item (conditioning), so its first row
    uses the same table row, position and conditioning row as row 0."""
    if world == 1:
        return case
    r0, r1 = shard_rows(world * case.rows, world, rank)
    period = max(case.seq_len, 1)
    if case.kind == "rope_pos":
        g = case.meta["grid"]
        period = g[0] * g[1] * g[2]
    if case.kind == "adaln":
        period = case.rows_per_cond
    if r0 % period:
        raise ValueError(f"{case.name}: shard start {r0} is not a multiple of {period}")
    meta = dict(case.meta, row_start=r0, batch_rows=world * case.rows)
    return Case(**{**case.__dict__, "rows": r1 - r0, "meta": meta})


def algorithmic_bytes(case: Case, per_row_tables: bool = False) -> int:
    """Bytes one call must move: read x, write y, read w (all bf16), plus the
    fp32 cos/sin tables at their literal size for the fused form, or the
    bf16 scale and shift for the AdaLN form.  GELU reads and writes one
    element per element; GEGLU reads two per output element and writes one
    (2 bytes each for bf16 and fp16, 4 for fp32)."""
    if case.kind in ("gelu", "rope_pos"):
        return (8 if case.dtype == "f32" else 4) * case.rows * case.hidden
    if case.kind == "geglu":
        return (12 if case.dtype == "f32" else 6) * case.rows * case.hidden
    e = 4 if case.dtype == "f32" else 2
    b = 2 * e * case.rows * case.hidden + (e * case.hidden if case.weight else 0)
    if case.kind == "add_norm":
        b += 2 * e * case.rows * case.hidden      # read the residual, write h
    if case.kind == "adaln":
        b += 2 * e * case.n_cond * case.hidden
    if case.mode is not None:
        P = case.head_dim // 2
        table_rows = case.rows if per_row_tables else case.seq_len
        b += 8 * table_rows * P
    return b
