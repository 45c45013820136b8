"""Benchmark: achieved HBM GB/s and us/call of bf16 RMSNorm / fused
RMSNorm+RoPE on GB300, through the C ABI of libltxk.so.

One step = one call per shape of the chosen workload.  The default,
``five_configs``, is the five configurations in one step: bf16 RMSNorm
[1x1024x2048], the shape sweep [2x1024x2048] .. [4x4096x3072], fused
RMSNorm + interleaved RoPE [2x4096, 32x128], fused RMSNorm + split-half RoPE
[6144, 32x64], and the bandwidth stress shapes [4x16384x4096],
[262143x2560], [65536x5120] (the largest problems, which dominate the
step's bytes and time).  Inputs are seeded, synthetic and resident in HBM
before the timed region; L2 is flushed (a 2x-L2 write, then a 2x-L2 read)
before every launch, outside the events.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ltxk|reference]

--impl reference times the fp64 CPU oracle on this host's cores on a bounded
row sample of the same workload (the method's plain definition, not a GPU
implementation).  Under torchrun (N > 1) the batch is N times the
workload's rows and every rank normalises its contiguous shard of the rows
(weak scaling: fixed rows per GPU, no data exchange); the time is the max
over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = ("achieved HBM GB/s (% of GB300 peak) for bf16 RMSNorm / "
          "RMSNorm+RoPE; µs/call")
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "rope_element_dit_gb300", "csrc")

WORKLOAD_TITLES = {
    "five_configs": "bf16 RMSNorm bandwidth stress [4x16384x4096], [262143x2560], "
                    "[65536x5120] (U(-4,4), eps 1e-5, seeds 7-9), timed in one step with "
                    "RMSNorm [1x1024x2048] (seed 0), the shape sweep [2x1024x2048], "
                    "[4x1024x2048], [2x4096x3072], [4x4096x3072] (1% x50 outliers, seeds "
                    "1-4), fused RMSNorm + interleaved RoPE [2x4096, 32x128] (seed 5) and "
                    "fused RMSNorm + split-half RoPE [6144, 32x64], 3-axis positions "
                    "(seed 6); w ~ N(1,0.1)",
    "sweep": "bf16 RMSNorm shape sweep [2x1024x2048], [4x1024x2048], "
             "[2x4096x3072], [4x4096x3072]; N(0,1) with 1% x50 outliers, "
             "w ~ N(1,0.1), eps 1e-6, seeds 1-4",
    "small": "bf16 RMSNorm [1x1024x2048], N(0,1), w ~ N(1,0.1), eps 1e-6, seed 0",
    "rope_interleaved": "fused RMSNorm + interleaved RoPE, x [2, 4096, 32x128], "
                        "fp32 cos/sin [4096, 64] (theta 1e4), seed 5",
    "rope_split": "fused RMSNorm + split-half RoPE, x [1, 6144, 32x64], 3-axis "
                  "positions 8x24x32, fp32 cos/sin [6144, 32], seed 6",
    "stress": "bf16 RMSNorm [4x16384x4096], [262143x2560], [65536x5120], "
              "U(-4,4), eps 1e-5, seeds 7-9",
    "adaln": "AdaLN-modulated RMSNorm norm(x)*(1+scale)+shift, x [2, 6144, 2048], "
             "no weight, scale/shift [2, 2048] ~ N(0, 0.5), seed 10",
    "add_norm": "fused residual add + RMSNorm, h = x + residual, y = RMSNorm(h), "
                "[4, 4096, 3072], x, residual ~ N(0,1), w ~ N(1,0.1), seed 11",
    "f16": "fp16 RMSNorm [4x4096x3072], N(0,1) with 1% x50 outliers, w ~ N(1,0.1), "
           "eps 1e-6, seed 14",
    "f32": "fp32 RMSNorm [4x4096x3072], N(0,1) with 1% x50 outliers, w ~ N(1,0.1), "
           "eps 1e-6, seed 15",
    "rope_pos_text": "standalone RoPE, angles from 1D positions on the device, x [2, 4096, "
                     "32 heads x 128] interleaved, theta 1e4, N(0,1), seed 16",
    "rope_pos_video": "standalone RoPE, angles from 3D positions (8x24x32, pairs 10/11/11) "
                      "on the device, x [1, 6144, 32 heads x 64] split-half, theta 1e4, seed 17",
    "gelu": "tanh-approximated GELU, x [2, 6144, 8192] (LTX-Video feed-forward inner "
            "width), N(0,1) with 1% x50 outliers, seed 12",
    "geglu": "GEGLU value * gelu_tanh(gate), x [2, 6144, 2x8192] -> [2, 6144, 8192], "
             "N(0,1) with 1% x50 outliers, seed 13",
    "gelu_f16": "fp16 tanh-approximated GELU, x [2, 6144, 8192], N(0,1) with 1% x50 "
                "outliers, seed 18",
    "gelu_f32": "fp32 tanh-approximated GELU, x [2, 6144, 8192], N(0,1) with 1% x50 "
                "outliers, seed 19",
    "geglu_f16": "fp16 GEGLU, x [2, 6144, 2x8192] -> [2, 6144, 8192], N(0,1) with 1% x50 "
                 "outliers, seed 20",
    "geglu_f32": "fp32 GEGLU, x [2, 6144, 2x8192] -> [2, 6144, 8192], N(0,1) with 1% x50 "
                 "outliers, seed 21",
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="five_configs", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--case", type=int, default=None,
                    help="run only this shape (index) of the workload, e.g. for a profiler "
                         "capture that should hold one shape on the device")
    ap.add_argument("--impl", default="ltxk", choices=["ltxk", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--path", default="auto", choices=["auto", "registers", "tma"],
                    help="kernel family for the vectorised cases")
    return ap.parse_args()


# ---------------------------------------------------------------- helpers --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# Rows [r0, r1) of a batch that rank `rank` of `world` normalises.
shard_rows = synth.shard_rows


def max_over_ranks(seconds, world, device=None):
    """The slowest rank's time (the job's time) via an all-reduce MAX."""
    if world == 1:
        return seconds
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbps(bytes_per_rank_step, steps, world, job_seconds):
    """Whole-job throughput: bytes all ranks moved / the job's time."""
    return world * bytes_per_rank_step * steps / job_seconds / 1e9


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)"


# The files that define each family of timed kernels and its launch
# configuration; traffic recorded by ncu stays valid while none of them changes.
KERNEL_SOURCES = {
    "rows": ("ltxk_kernels.cuh", "ltxk_instances.cuh", "ltxk_launch.h", "ltxk_abi.cu",
             "ltxk_rows_plain.cu", "ltxk_rows_interleaved.cu", "ltxk_rows_split.cu",
             "ltxk_rows_adaln.cu", "ltxk_rows_addnorm.cu"),
    "gelu": ("ltxk_kernels.cuh", "ltxk_launch.h", "ltxk_gelu.cu"),
    "rope": ("ltxk_kernels.cuh", "ltxk_launch.h", "ltxk_rope.cu"),
}


def kernel_family(kernel):
    if kernel.startswith(("gelu", "geglu")):
        return "gelu"
    return "rope" if kernel.startswith("rope_kernel") else "rows"


_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def code_text(src: str) -> str:
    """The code of a C++/CUDA source without its comments and with runs of
    whitespace collapsed, so that a change to a comment alone keeps the
    digest (string literals in these sources hold no comment markers)."""
    return " ".join(_COMMENT.sub(" ", src).split())


def source_digest(family="rows", read=None):
    """Digest of the code (comments and layout aside) of a kernel family's
    sources.  ``read(name)`` returns a source's text (default: the file)."""
    h = hashlib.sha256()
    for fn in KERNEL_SOURCES[family]:
        if read is None:
            with open(os.path.join(CSRC, fn), encoding="utf-8") as f:
                text = f.read()
        else:
            text = read(fn)
        h.update(fn.encode() + b"\0" + code_text(text).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, case, digest):
    """DRAM bytes per launch of one case (shape) from the committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split("\t")
        if len(parts) >= 4 and parts[0] == kernel and parts[1] == case \
                and parts[2] == digest:
            return int(parts[3])
    return None


class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""
    QUERY = ("timestamp,index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id):
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            f = [s.strip() for s in line.split(",")]
            if len(f) < 11:
                continue
            if self.bus_id and self.bus_id not in f[2].lower() and \
                    f[2].lower()[-12:] != self.bus_id[-12:]:
                continue
            rows.append((ts, f))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = [r for r in rows if t0 <= r[0] <= t1 + 0.25] or \
            sorted(rows, key=lambda r: abs(r[0] - (t0 + t1) / 2))[:3]
        sm = [float(f[3]) for _, f in inside if f[3].replace(".", "").isdigit()]
        mx = [float(f[4]) for _, f in inside if f[4].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for _, f in inside:
            for name, v in zip(names, f[7:11]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "power_w_max": max((float(f[5]) for _, f in inside
                                    if f[5].replace(".", "").isdigit()), default=None)}


# ---------------------------------------------------------- oracle timing --

def cpu_oracle_time(cases, inputs, row_frac, threads):
    """Run the oracle over the first ceil(row_frac * rows) rows of every case;
    returns (seconds, algorithmic bytes)."""
    import oracle
    t = 0.0
    b = 0
    for c, inp in zip(cases, inputs):
        r = max(1, math.ceil(c.rows * row_frac))
        x = inp["x"][:r]
        t0 = time.perf_counter()
        if c.kind == "rope_pos":
            oracle.rope(x, c.heads, c.head_dim, c.mode, tuple(c.meta["grid"]),
                        tuple(c.meta["pairs"]), c.meta["theta"], threads=threads)
        elif c.kind == "gelu":
            oracle.gelu_tanh(x, threads=threads)
        elif c.kind == "geglu":
            oracle.geglu(x, threads=threads)
        elif c.kind == "add_norm":
            oracle.add_rms_norm(x, inp["res"][:r], inp["w"], c.eps, threads=threads)
        elif c.kind == "adaln":
            oracle.rms_norm_adaln(x, inp["w"], inp["scale"], inp["shift"], c.eps,
                                  rows_per_cond=c.rows_per_cond, threads=threads)
        elif c.mode is None:
            oracle.rms_norm(x, inp["w"], c.eps, threads=threads)
        else:
            oracle.rms_norm_rope(x, inp["w"], inp["cos"], inp["sin"], c.heads, c.head_dim,
                                 c.mode, c.eps, table_rows=c.seq_len, threads=threads)
        t += time.perf_counter() - t0
        if c.kind in ("gelu", "geglu", "rope_pos"):
            b += (3 if c.kind == "geglu" else 2) * inp["x"].dtype.itemsize * r * c.hidden
            continue
        e = inp["x"].dtype.itemsize
        b += 2 * e * r * c.hidden + (e * c.hidden if inp["w"] is not None else 0) + (
            8 * min(r, c.seq_len) * (c.head_dim // 2) if c.mode is not None else 0) + (
            2 * e * (-(-r // c.rows_per_cond)) * c.hidden if c.kind == "adaln" else 0) + (
            2 * e * r * c.hidden if c.kind == "add_norm" else 0)
    return t, b


def cpu_baseline(cases, inputs, seconds):
    threads = os.cpu_count() or 1
    # calibrate on a 1% row sample, then size the sample to ~`seconds`
    t, _ = cpu_oracle_time(cases, inputs, 0.01, threads)
    frac = min(1.0, max(0.01, 0.01 * seconds / max(t, 1e-6)))
    reps = 1
    if frac >= 1.0:
        t_full, _ = cpu_oracle_time(cases, inputs, 1.0, threads)
        reps = max(1, math.ceil(seconds / max(t_full, 1e-6)))   # at least `seconds`
    tot_t, tot_b = 0.0, 0
    for _ in range(reps):
        tt, bb = cpu_oracle_time(cases, inputs, frac, threads)
        tot_t += tt
        tot_b += bb
    sample = (f"fp64 C oracle, {threads} threads over row blocks, first "
              f"{frac * 100:.1f}% of the rows of every shape"
              + (f", {reps} repetitions" if reps > 1 else "")
              + f", {tot_t:.1f} s")
    # the same oracle on one thread, over a sample sized to about a quarter of
    # the time budget
    t1, _ = cpu_oracle_time(cases, inputs, 0.001, 1)
    frac1 = min(1.0, max(0.001, 0.001 * 0.25 * seconds / max(t1, 1e-6)))
    st, sb = cpu_oracle_time(cases, inputs, frac1, 1)
    return {"value": round(tot_b / tot_t / 1e9, 3), "unit": UNIT, "cores": threads,
            "kind": "oracle", "sample": sample,
            "single_thread": {"value": round(sb / st / 1e9, 4), "unit": UNIT, "cores": 1,
                              "sample": f"first {frac1 * 100:.2f}% of the rows of every "
                                        f"shape, {st:.1f} s"}}


def run_reference(args, cases, inputs, world, rank):
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    budget = 120.0      # seconds of oracle work for the whole run
    t1, _ = cpu_oracle_time(cases, inputs, 0.01, threads)
    per_step = budget / max(1, args.steps + args.warmup)
    frac = min(1.0, max(1e-4, 0.01 * per_step / max(t1, 1e-9)))
    for _ in range(args.warmup):
        cpu_oracle_time(cases, inputs, frac, threads)
    tt = 0.0
    bb = 0
    for _ in range(args.steps):
        t, b = cpu_oracle_time(cases, inputs, frac, threads)
        tt += t
        bb += b
    value = bb / tt / 1e9
    sample = (f"fp64 C oracle on {threads} host threads; each step the first "
              f"{frac * 100:.3g}% of the rows of every shape")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tt / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_keys(args, cases) | {"row_fraction": frac},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def config_keys(args, cases):
    """The keys that name the workload, the same in both arms."""
    d = {"workload": WORKLOAD_TITLES[args.workload], "name": args.workload, "case": args.case,
         "shapes": [c.name for c in cases]}
    if args.workload == "five_configs":
        d["headline"] = WORKLOAD_TITLES["stress"]
    return d


# ------------------------------------------------------------- GPU timing --

DTYPE_CODES = {"bf16": 0, "f16": 1, "f32": 2}


def kernel_name(plan, mode, dtype="bf16"):
    """Kernel instance name as ncu prints it; mode None = plain, 0/1 = RoPE
    pairing, 3 = AdaLN, 4 = residual add + RMSNorm; the last template
    argument is the element format (0 bf16, 1 fp16, 2 fp32)."""
    import rope_element_dit_gb300 as L
    km = 0 if mode is None else {0: 1, 1: 2, 3: 3, 4: 4}[mode]
    f = DTYPE_CODES[dtype]
    if plan.kernel == L.KERNEL_ROWS_VEC:
        return f"rows_vec_kernel<{km}, {plan.group_warps}, {plan.vec_per_lane}, {f}>"
    if plan.kernel == L.KERNEL_ROWS_TMA:
        return f"rows_tma_kernel<{km}, {plan.vec_per_lane}>"
    return f"rows_elem_kernel<{km}, {f}>"


def _tensor(a):
    """torch view of a generated array (bf16 bit patterns travel as int16)."""
    import torch
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)


def run_ltxk(args, cases, inputs, world, rank, local):
    import torch
    import rope_element_dit_gb300 as L

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    props = torch.cuda.get_device_properties(dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream

    # resident inputs and outputs
    dev_bufs = []
    for c, inp in zip(cases, inputs):
        xt = _tensor(inp["x"])
        d = {"x": xt.to(dev),
             "w": None if inp["w"] is None else _tensor(inp["w"]).to(dev),
             "y": torch.empty(c.rows * c.hidden, dtype=xt.dtype, device=dev)}
        if c.kind == "add_norm":
            d["res"] = _tensor(inp["res"]).to(dev)
            d["h"] = torch.empty(c.rows * c.hidden, dtype=xt.dtype, device=dev)
        if c.kind == "adaln":
            d["scale"] = _tensor(inp["scale"]).to(dev)
            d["shift"] = _tensor(inp["shift"]).to(dev)
        if c.kind == "rope":
            d["cos"] = torch.from_numpy(inp["cos"]).to(dev)
            d["sin"] = torch.from_numpy(inp["sin"]).to(dev)
        dev_bufs.append(d)

    def call_args(i, x=None, y=None, res=None, h=None):
        c, d = cases[i], dev_bufs[i]
        x = d["x"] if x is None else x
        d = dict(d, y=d["y"] if y is None else y)
        if c.kind == "add_norm":
            d = dict(d, res=d["res"] if res is None else res, h=d["h"] if h is None else h)
        wp = None if d["w"] is None else d["w"].data_ptr()
        if c.kind == "rope_pos":
            return L.ltxk_rope, (d["y"].data_ptr(), x.data_ptr(), c.rows, c.heads, c.head_dim,
                                 c.mode, *c.meta["grid"], *c.meta["pairs"], c.meta["theta"],
                                 DTYPE_CODES[c.dtype], sptr)
        if c.kind == "gelu":
            return L.ltxk_gelu_tanh_dt, (d["y"].data_ptr(), x.data_ptr(), c.rows * c.hidden,
                                         DTYPE_CODES[c.dtype], sptr)
        if c.kind == "geglu":
            return L.ltxk_geglu_dt, (d["y"].data_ptr(), x.data_ptr(), c.rows, c.hidden,
                                     DTYPE_CODES[c.dtype], sptr)
        if c.kind == "add_norm":
            return L.ltxk_add_rms_norm, (d["y"].data_ptr(), d["h"].data_ptr(), x.data_ptr(),
                                         d["res"].data_ptr(), wp, c.rows, c.hidden, c.eps,
                                         sptr)
        if c.kind == "adaln":
            return L.ltxk_rms_norm_adaln, (
                d["y"].data_ptr(), x.data_ptr(), wp, d["scale"].data_ptr(),
                d["shift"].data_ptr(), c.rows, c.hidden, c.rows_per_cond, c.eps, sptr)
        if c.mode is None and c.dtype != "bf16":
            return L.ltxk_rms_norm_dt, (d["y"].data_ptr(), x.data_ptr(), wp, c.rows, c.hidden,
                                        c.eps, DTYPE_CODES[c.dtype], sptr)
        if c.mode is None:
            return L.ltxk_rms_norm, (d["y"].data_ptr(), x.data_ptr(), wp,
                                     c.rows, c.hidden, c.eps, sptr)
        return L.ltxk_rms_norm_rope_seq, (
            d["y"].data_ptr(), x.data_ptr(), wp, d["cos"].data_ptr(),
            d["sin"].data_ptr(), c.rows, c.heads, c.head_dim, c.mode, c.eps, c.seq_len, sptr)

    # prebuilt calls keep the host side of a launch to one ctypes call
    calls = [call_args(i) for i in range(len(cases))]

    def launch(i, x=None, y=None, res=None, h=None):
        fn, a = calls[i] if x is None and y is None else call_args(i, x, y, res, h)
        st = fn(*a)
        if st != L.OK:
            raise L.LtxkError(st, "bench launch")

    L.ltxk_set_path({"auto": L.PATH_AUTO, "registers": L.PATH_REGISTERS,
                     "tma": L.PATH_TMA}[args.path])
    l2 = getattr(props, "L2_cache_size", 0) or (126 << 20)
    flush_w = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(2 * l2 // 4, dtype=torch.float32, device=dev)

    def flush_l2(i):
        # write 2x L2 (evicts everything), then read another 2x L2 (a float32
        # sum reads it in place) so that the written lines are written back
        # here and L2 is left clean and cold
        flush_w.fill_(i & 0xFF)
        flush_r.sum()

    n = len(cases)
    bytes_per_launch = [synth.algorithmic_bytes(c) for c in cases]
    bytes_per_step = sum(bytes_per_launch)
    plans = []
    for c in cases:
        if c.kind in ("gelu", "geglu"):
            f = DTYPE_CODES[c.dtype]
            if c.dtype == "f32":
                plans.append("gelu_chunk_kernel" if c.kind == "gelu" else
                             "geglu_chunk_kernel<unsigned int>")
            else:
                plans.append(f"gelu_vec_kernel<{f}>" if c.kind == "gelu" else
                             f"geglu_vec_kernel<unsigned int, {f}>")
            continue
        if c.kind == "rope_pos":
            # the library's block rule: 64 threads when a row's 16-byte units
            # (lo/hi pairs for split-half) fit one pass of 64 threads
            units = c.hidden // 8 if c.mode == 0 else c.heads * (c.head_dim // 16)
            per_thread = (4 if c.mode == 0 else 2) // (2 if c.dtype == "f32" else 1)
            block = 64 if units <= 64 * per_thread else 128
            plans.append(f"rope_kernel<{1 if c.mode == 0 else 2}, {DTYPE_CODES[c.dtype]}, true, "
                         f"{block}>")
            continue
        op = {"norm": L.OP_RMS_NORM, "rope": L.OP_RMS_NORM_ROPE,
              "adaln": L.OP_RMS_NORM_ADALN, "add_norm": L.OP_ADD_RMS_NORM}[c.kind]
        st, p = L.ltxk_plan_launch_dt(op, DTYPE_CODES[c.dtype], c.rows, c.hidden, c.head_dim,
                                      c.mode or 0, True)
        plans.append(kernel_name(p, {"adaln": 3, "add_norm": 4}.get(c.kind, c.mode), c.dtype))

    for i in range(args.warmup):
        flush_l2(i)
        for j in range(n):
            launch(j)
    torch.cuda.synchronize()

    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)] for _ in range(args.steps)]
    # A GPU-side spin before each step's first event gives the host time to
    # queue the whole step, so no launch latency of the host lands inside the
    # events (the spin, like the L2 flush, is outside them).
    t_host = time.perf_counter()
    for i in range(20):
        for j in range(n):
            launch(j)
    torch.cuda.synchronize()
    host_per_step = (time.perf_counter() - t_host) / 20
    spin_cycles = int(min(2e6, max(1e5, 4 * host_per_step / n * 2.0e9)))
    try:
        bus = "{:08X}:{:02X}:{:02X}.0".format(props.pci_domain_id, props.pci_bus_id,
                                              props.pci_device_id)
    except AttributeError:
        bus = None
    sampler = ClockSampler(bus)
    if not args.no_clocks:
        sampler.start()
        time.sleep(0.6)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        for j in range(n):
            flush_l2(i * n + j)
            torch.cuda._sleep(spin_cycles)
            ev[i][j][0].record(stream)
            launch(j)
            ev[i][j][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    if not args.no_clocks:
        time.sleep(0.3)
        sampler.stop()

    per_launch = np.array([[ev[i][j][0].elapsed_time(ev[i][j][1]) for j in range(n)]
                           for i in range(args.steps)], dtype=np.float64)   # ms
    step_ms = per_launch.sum(axis=1)
    total_s = max_over_ranks(step_ms.sum() / 1e3, world, dev)
    value = aggregate_gbps(bytes_per_step, args.steps, world, total_s)

    # dominant kernel: the kernel instance with the largest share of time
    by_kernel = {}
    peak, peak_kind = measured_peak()
    per_shape = []
    for j, c in enumerate(cases):
        us = per_launch[:, j] * 1e3
        med = float(np.median(us))
        mean = float(us.mean())
        dram = recorded_traffic(plans[j], c.name, source_digest(kernel_family(plans[j])))
        k = by_kernel.setdefault(plans[j], {"bytes": 0, "ms": 0.0, "launches": 0, "dram": 0,
                                            "dram_known": True})
        k["bytes"] += bytes_per_launch[j] * args.steps
        k["ms"] += per_launch[:, j].sum()
        k["launches"] += args.steps
        if dram is None:
            k["dram_known"] = False
        else:
            k["dram"] += dram * args.steps
        per_shape.append({
            "case": c.name, "kernel": plans[j], "bytes": bytes_per_launch[j],
            "us_mean": round(mean, 3), "gbps_mean": round(bytes_per_launch[j] / mean / 1e3, 1),
            "us_median": round(med, 3), "us_p10": round(float(np.percentile(us, 10)), 3),
            "us_p90": round(float(np.percentile(us, 90)), 3),
            "gbps_median": round(bytes_per_launch[j] / med / 1e3, 1),
            # CUDA event timestamps advance in steps of about 1 us on this
            # device, so a median of a short kernel is one of those steps;
            # the mean over the launches is not quantised that way
            "frac_of_peak": round(bytes_per_launch[j] / mean / 1e3 / peak, 4),
            # DRAM bytes of one ncu capture of this shape over the live time
            "dram_bytes": dram,
            "dram_frac_of_peak": None if dram is None else round(dram / mean / 1e3 / peak, 4)})
    dom_name, dom = max(by_kernel.items(), key=lambda kv: kv[1]["ms"])
    achieved = dom["bytes"] / (dom["ms"] / 1e3) / 1e9
    digest = source_digest(kernel_family(dom_name))
    traffic = dom["dram"] // dom["launches"] if dom["dram_known"] else None
    achieved_dram = None if traffic is None else traffic * dom["launches"] / (dom["ms"] / 1e3) / 1e9

    # e2e: host (pinned) x -> host y through the public API.  bf16 RMSNorm
    # goes through the host call ltxk_rms_norm_host; the other workloads call
    # their entry point on the pinned tensors.  Either way the kernel reads x
    # and writes y across the host link itself (zero-copy).
    e2e = None
    if not args.no_e2e:
        hx = [_tensor(inp["x"]).reshape(-1).pin_memory() for inp in inputs]
        hy = [torch.empty(c.rows * c.hidden, dtype=d["y"].dtype).pin_memory()
              for c, d in zip(cases, dev_bufs)]
        # the residual add streams its second input and second output (the
        # new residual stream h) across the host link as well
        hres = [_tensor(inp["res"]).reshape(-1).pin_memory() if c.kind == "add_norm" else None
                for c, inp in zip(cases, inputs)]
        hh = [torch.empty_like(hy[j]).pin_memory() if c.kind == "add_norm" else None
              for j, c in enumerate(cases)]
        h2d = sum(h.numel() * h.element_size() for h in hx + hres if h is not None)
        d2h = sum(h.numel() * h.element_size() for h in hy + hh if h is not None)
        # bf16 RMSNorm shapes go through the host call, the others through
        # their entry point on the pinned tensors
        host_call = [c.kind == "norm" and c.dtype == "bf16" for c in cases]
        pstreams = [torch.cuda.Stream(dev) for _ in range(3)]
        handles = [ps.cuda_stream for ps in pstreams]
        # one staging buffer per host-call shape: calls on rotated streams
        # never share slots, whichever branch (zero-copy or staged) a call takes
        staging = [torch.empty(3 * (16 << 20), dtype=torch.uint8, device=dev) if hc else None
                   for hc in host_call]
        e_ms = []
        for i in range(args.e2e_steps + 3):
            flush_l2(i)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for ps in pstreams:
                ps.wait_stream(stream)
            for j, c in enumerate(cases):
                if not host_call[j]:
                    # the call itself on the pinned host tensors: the kernel
                    # reads x and writes y across the host link (zero-copy)
                    launch(j, x=hx[j], y=hy[j], res=hres[j], h=hh[j])
                    continue
                wp = None if dev_bufs[j]["w"] is None else dev_bufs[j]["w"].data_ptr()
                # independent shapes start on different streams, so their
                # fixed latencies overlap
                rot = handles[j % len(handles):] + handles[:j % len(handles)]
                st = L.ltxk_rms_norm_host(hy[j].data_ptr(), hx[j].data_ptr(), wp, c.rows,
                                          c.hidden, c.eps, staging[j].data_ptr(),
                                          staging[j].numel(), rot, len(rot))
                if st != L.OK:
                    raise L.LtxkError(st, "bench e2e")
            for ps in pstreams:
                stream.wait_stream(ps)
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                e_ms.append(e0.elapsed_time(e1))
        e2e_s = max_over_ranks(sum(e_ms) / 1e3, world, dev)
        notes = []
        if any(host_call):
            notes.append("bf16 RMSNorm shapes: ltxk_rms_norm_host on pinned host x and y, one "
                         "kernel reads x and writes y across the host link (NVLink-C2C on "
                         "GB300, zero-copy), the shapes start on three streams in turn")
        if not all(host_call):
            notes.append("other shapes: the ltxk call on pinned host x and y (and, for the "
                         "residual add, residual and h), the kernel reads and writes them "
                         "across the host link (zero-copy)")
        notes.append("weight, tables and conditioning vectors resident")
        e2e = {"value": round(aggregate_gbps(bytes_per_step, len(e_ms), world, e2e_s), 2),
               "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_s / len(e_ms) * 1e3, 4), "note": "; ".join(notes)}

    clocks = sampler.summary(t0, t1) if not args.no_clocks else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cases, inputs, args.cpu_seconds)

    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(float(step_ms.mean()), 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "io_dtype": cases[0].dtype, "data": "synthetic",
        "config": config_keys(args, cases) | {
                   "timing": "CUDA events around each launch on the launching stream; "
                             "a GPU spin before each launch keeps host launch latency "
                             "out of the events",
                   "host_us_per_step": round(host_per_step * 1e6, 1),
                   "l2": f"flushed before every launch, outside the timed events: a "
                         f"{2 * l2 >> 20} MiB write, then a {2 * l2 >> 20} MiB read of "
                         "another buffer (cold and clean L2 at kernel start)",
                   "path": args.path,
                   "bytes_per_step": bytes_per_step, "per_shape": per_shape,
                   "parallelism": (f"rows of one batch of {world} x the workload's rows "
                                   f"split over {world} GPUs, no exchange"
                                   if world > 1 else "1 GPU")},
        "frac_of_peak": round(value / world / peak, 4),
        "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     # the same launches' DRAM bytes (ncu) over their live time
                     "achieved_dram": None if achieved_dram is None else round(achieved_dram, 1),
                     "frac_dram": None if achieved_dram is None else round(achieved_dram / peak, 4),
                     "algorithmic_bytes_per_launch": int(dom["bytes"] / dom["launches"]),
                     "launches": dom["launches"], "source_digest": digest},
        "e2e": e2e, "clocks": clocks, "cpu_baseline": cpu,
        "gpu_launches": n * args.steps,
        "device": props.name,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_env()
    cases = synth.WORKLOADS[args.workload]
    if args.case is not None:
        if not 0 <= args.case < len(cases):
            raise SystemExit(f"--case must be in [0, {len(cases)})")
        cases = [cases[args.case]]
    if args.impl == "ltxk" and world > 1:
        cases = [synth.shard_case(c, world, rank) for c in cases]
    inputs = [synth.make_inputs(c) for c in cases]
    if args.impl == "reference":
        run_reference(args, cases, inputs, world, rank)
        return
    run_ltxk(args, cases, inputs, world, rank, local)


if __name__ == "__main__":
    main()
