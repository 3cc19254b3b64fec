"""Build libmegamoe.so in-tree for sm_103a (nvcc; translation units in parallel)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmegamoe.so")
SOURCES = ["api.cu", "route.cu", "megamoe.cu", "quant.cu", "noalloc.cu"]
HEADERS = ["common.cuh", "numerics.cuh"]
ARCH = "103a"


def _flags():
    return [f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}", "-O3", "-lineinfo", "-std=c++17",
            "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def _stale(out, deps):
    return not os.path.exists(out) or os.path.getmtime(out) < max(os.path.getmtime(d) for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(HERE, "..", "include", "megamoe.h")]
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            jobs.append((s, o))

    def compile_one(job):
        s, o = job
        tmp = o + f".tmp{os.getpid()}"
        r = subprocess.run(["nvcc", *_flags(), "-c", s, "-o", tmp], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {s}:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, o)
        return s, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for s, log in ex.map(compile_one, jobs):
            if verbose:
                print(f"== {os.path.basename(s)}\n{log}")
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["nvcc", f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}", "-shared",
                               "-Xcompiler", "-fPIC", *objs, "-o", tmp])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True)
