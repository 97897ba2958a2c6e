"""Build libspecverify.so for sm_103a with nvcc (one -gencode, translation
units compiled in parallel, CUDA runtime linked statically)."""

from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libspecverify.so")
SOURCES = ["api.cu", "linear.cu", "rows_topp.cu", "decide.cu", "draw_stream.cu", "tree.cu", "compact.cu", "sample_rows.cu"]
# threads per CTA of the row-level kernels in each unit (see common.cuh)
CTA_THREADS = {"decide.cu": 512, "tree.cu": 512, "sample_rows.cu": 512}
# units whose CTAs hold a copy warp beside the row threads: row barriers are
# named barriers over the row threads only
NAMED_ROW_BARRIER = {"rows_topp.cu", "draw_stream.cu"}
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libspecverify needs the CUDA toolkit to build")


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src] + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "specverify.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile every translation unit and link libspecverify.so; returns its path."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, s):
            nt = [f"-DSV_NT={CTA_THREADS[src]}"] if src in CTA_THREADS else []
            if src in NAMED_ROW_BARRIER:
                nt.append("-DSV_ROW_BARRIER_NAMED")
            jobs.append([nvcc, *ARCH, *FLAGS, *nt, *extra_flags, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        return r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        for out in ex.map(run, jobs):
            if verbose and out.strip():
                print(out)
    # relink also when an earlier link failed after its objects were built
    if force or jobs or not os.path.exists(LIB) or any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        run([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
