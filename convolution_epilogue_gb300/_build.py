"""Builds libfusedconv.so in-tree with nvcc (sm_103a only).

Every translation unit under csrc/ is compiled in parallel to an object
file, then linked into convolution_epilogue_gb300/_build/libfusedconv.so.
Objects are rebuilt when their source or any header is newer.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libfusedconv.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _headers():
    return (glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def build(verbose: bool = False, force: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    newest_hdr = max((os.path.getmtime(h) for h in _headers()), default=0)
    jobs = []
    objs = []
    for s in srcs:
        o = os.path.join(OUT, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if (force or not os.path.exists(o) or os.path.getmtime(o) < os.path.getmtime(s)
                or os.path.getmtime(o) < newest_hdr):
            jobs.append((s, o))

    def compile_one(job):
        s, o = job
        cmd = [nvcc()] + ARCH + NVCC_FLAGS + ["-I", INCLUDE, "-c", s, "-o", o + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {s}:\n{r.stdout}\n{r.stderr}")
        os.replace(o + ".tmp", o)
        return r.stderr

    if jobs:
        with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            for msg in ex.map(compile_one, jobs):
                if verbose and msg:
                    print(msg)
    if (force or jobs or not os.path.exists(LIB)
            or any(os.path.getmtime(LIB) < os.path.getmtime(o) for o in objs)):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
