"""Build libltxk.so in-tree with nvcc for sm_103a (GB300).

The translation units compile in parallel; one ``-gencode`` target only.
``python rope_element_dit_gb300/build.py`` runs it from the command line (not
``-m``: importing the package loads the library this script builds).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libltxk.so")

SOURCES = ["ltxk_abi.cu", "ltxk_noalloc.cu", "ltxk_pipeline.cu", "ltxk_gelu.cu", "ltxk_rope.cu"]
# Row-kernel instance files, compiled once per element format (LTXK_FMT:
# 0 bf16, 1 fp16, 2 fp32).
ROW_SOURCES = ["ltxk_rows_plain.cu", "ltxk_rows_interleaved.cu", "ltxk_rows_split.cu",
               "ltxk_rows_adaln.cu", "ltxk_rows_addnorm.cu"]
FORMATS = {0: "bf16", 1: "f16", 2: "f32"}
HEADERS = ["ltxk_kernels.cuh", "ltxk_instances.cuh", "ltxk_launch.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libltxk")
    return cand


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(),
          out_dir: str | None = None) -> str:
    """Compile (only what is stale) and link libltxk.so.  ``extra_flags`` are
    added to every nvcc compile; ``out_dir`` puts the objects and the library
    in another directory (for building variants side by side)."""
    nvcc = _nvcc()
    obj_dir = OBJ_DIR if out_dir is None else os.path.join(out_dir, "_build")
    lib = LIB if out_dir is None else os.path.join(out_dir, "libltxk.so")
    os.makedirs(obj_dir, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "ltxk.h")]
    objs = []
    jobs = []
    units = [(src, src.replace(".cu", ".o"), []) for src in SOURCES]
    units += [(src, src.replace(".cu", f".{name}.o"), [f"-DLTXK_FMT={fmt}"])
              for src in ROW_SOURCES for fmt, name in FORMATS.items()]
    for src, obj, defs in units:
        s = os.path.join(CSRC, src)
        o = os.path.join(obj_dir, obj)
        objs.append(o)
        if force or _stale(o, [s] + headers):
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, *defs, *extra_flags, "-c", s, "-o", o]
            jobs.append(cmd)

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)

    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        list(ex.map(run, jobs))

    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", "-rpath," + _cuda_lib_dir(nvcc)]
        run(cmd)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
