"""Compile the CUDA library in-tree for sm_103a (nvcc only, no cmake).

build() makes libonebit_adam.so.  build(checked=True) makes libonebit_adam_checked.so, the same
library compiled with -DONEBIT_CHECKS: every kernel checks its units of work against its buffers
before touching them, skips any that fail and reports them through onebit_adam_get_status().  The
package loads the checked library when the environment variable ONEBIT_LIBRARY is "checked".
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libonebit_adam.so")
LIB_CHECKED = os.path.join(HERE, "libonebit_adam_checked.so")
BUILD_DIR = os.path.join(HERE, "_build")

SOURCES = ["onebit_adam.cu", "onebit_noalloc.cu"]
HEADERS = ["onebit_kernels.cuh", os.path.join("..", "..", "include", "onebit_adam.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "--fmad=false",            # no contraction: the fp32 op order must match the method's formulas
    "-prec-div=true", "-prec-sqrt=true",
    "-Xcompiler", "-fPIC,-O2",
    "-I", os.path.join(ROOT, "include"),
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    lib = LIB_CHECKED if checked else LIB
    bdir = os.path.join(BUILD_DIR, "checked") if checked else BUILD_DIR
    flags = [*NVCC_FLAGS, "-DONEBIT_CHECKS"] if checked else NVCC_FLAGS
    os.makedirs(bdir, exist_ok=True)
    hdrs = [os.path.normpath(os.path.join(CSRC, h)) for h in HEADERS]
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s, *hdrs, __file__]):
            jobs.append([nvcc(), *flags, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        if verbose:
            print(r.stdout + r.stderr)

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        run([nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
