"""Host logic of bench.py that needs no GPU: the code digest that keys the
committed ncu traffic figures, and the lookup of those figures."""
import os

import bench


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


def test_recorded_traffic_is_keyed_by_kernel_workload_and_digest():
    lines = [l.split("\t") for l in open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.txt"))
             if l.strip() and not l.startswith("#")]
    assert lines
    k, w, d, b = lines[0]
    assert bench.recorded_traffic(k, w, d) == int(b)
    assert bench.recorded_traffic(k, w, "0" * 16) is None
    assert bench.recorded_traffic(k, "no_such_workload", d) is None
