"""Host logic of bench.py that needs no GPU: the code digest that keys the
committed ncu traffic figures, the lookup of those figures, the default
workload, the keys that name it in both arms, and the row shards of the
multi-GPU mode."""
import argparse
import os

import numpy as np

import bench
import synth


def test_digest_ignores_comments_and_layout():
    src = "int f(int a) {\n  return a + 1;  // one more\n}\n/* block\n comment */\n"
    same = "int f(int a) { return a + 1; }\n"
    assert bench.code_text(src) == bench.code_text(same)
    texts = {"a.cu": src}
    fam = ("a.cu",)
    old = bench.KERNEL_SOURCES.get("test")
    bench.KERNEL_SOURCES["test"] = fam
    try:
        d1 = bench.source_digest("test", read=lambda fn: texts[fn])
        texts["a.cu"] = src.replace("// one more", "// the successor")
        assert bench.source_digest("test", read=lambda fn: texts[fn]) == d1
        texts["a.cu"] = src.replace("a + 1", "a + 2")
        assert bench.source_digest("test", read=lambda fn: texts[fn]) != d1
    finally:
        if old is None:
            del bench.KERNEL_SOURCES["test"]
        else:
            bench.KERNEL_SOURCES["test"] = old


def test_digest_reads_the_committed_sources():
    for fam, files in bench.KERNEL_SOURCES.items():
        for fn in files:
            assert os.path.exists(os.path.join(bench.CSRC, fn)), fn
        assert len(bench.source_digest(fam)) == 16


def test_recorded_traffic_is_keyed_by_kernel_case_and_digest():
    lines = [l.split("\t") for l in open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.txt"))
             if l.strip() and not l.startswith("#")]
    assert lines
    cases = {c.name for cs in synth.WORKLOADS.values() for c in cs}
    for k, case, d, b in lines:
        assert case in cases, case
        assert bench.recorded_traffic(k, case, d) == int(b)
    k, case, d, b = lines[0]
    assert bench.recorded_traffic(k, case, "0" * 16) is None
    assert bench.recorded_traffic(k, "no_such_case", d) is None


def test_default_workload_is_the_five_configurations():
    ap_default = [a for a in open(os.path.join(bench.ROOT, "bench.py"))
                  if 'add_argument("--workload"' in a]
    assert ap_default and 'default="five_configs"' in ap_default[0]
    names = [c.name for c in synth.WORKLOADS["five_configs"]]
    for wl in ("small", "sweep", "rope_interleaved", "rope_split", "stress"):
        for c in synth.WORKLOADS[wl]:
            assert c.name in names
    assert len(names) == 10


def test_both_arms_name_the_workload_with_the_same_keys():
    args = argparse.Namespace(workload="five_configs", case=None)
    cases = synth.WORKLOADS["five_configs"]
    k = bench.config_keys(args, cases)
    assert {"workload", "name", "case", "shapes", "headline"} <= set(k)
    assert k["headline"] == bench.WORKLOAD_TITLES["stress"]
    assert bench.config_keys(args, cases) == k


def test_shards_are_rows_of_one_batch():
    # every rank's shard is a contiguous slice of the batch of world x rows,
    # generated alone from the counter-based streams
    for wl in ("sweep", "adaln", "add_norm"):
        c = synth.WORKLOADS[wl][0]
        c = synth.Case(**{**c.__dict__, "rows": 12 if wl != "adaln" else 12,
                          "rows_per_cond": 6 if wl == "adaln" else 0})
        for world in (2, 3):
            whole = synth.Case(**{**c.__dict__, "rows": world * c.rows})
            full = synth.make_inputs(whole)
            parts = [synth.make_inputs(synth.shard_case(c, world, r)) for r in range(world)]
            assert np.array_equal(np.concatenate([p["x"] for p in parts]), full["x"])
            if wl == "add_norm":
                assert np.array_equal(np.concatenate([p["res"] for p in parts]), full["res"])
            if wl == "adaln":
                assert np.array_equal(np.concatenate([p["scale"] for p in parts]), full["scale"])
                assert np.array_equal(np.concatenate([p["shift"] for p in parts]), full["shift"])
    # the fused forms' shards start at a whole sequence: same tables
    c = synth.WORKLOADS["rope_interleaved"][0]
    s = synth.shard_case(c, 2, 1)
    assert s.rows == c.rows and s.meta["row_start"] % c.seq_len == 0
    assert synth.shard_case(c, 1, 0) is c
