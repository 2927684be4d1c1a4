"""The checked build on the host (no GPU): the library compiled with -DONEBIT_CHECKS builds for sm_103a
and exports every call the header declares; in normal builds the checks leave no trace in the
kernels (the preprocessed source holds none of them); and the kernel names its bounds report uses
follow the header's kernel enum."""
import os
import re
import subprocess

import ctypes
import pytest

import communication_compressed_optimizer_compress_gb300 as ob
from communication_compressed_optimizer_compress_gb300 import _build
from test_abi_host import _declared

CSRC = os.path.join(_build.HERE, "csrc")


def test_checked_library_builds_and_exports_every_symbol():
    lib = _build.build(checked=True)
    assert os.path.basename(lib) == "libonebit_adam_checked.so"
    L = ctypes.CDLL(lib)
    missing = [n for n in _declared() if not hasattr(L, n)]
    assert not missing, missing


def _preprocessed(*defines):
    r = subprocess.run([_build.nvcc(), "-E", "-x", "cu", "-std=c++17", "-I", os.path.join(_build.ROOT, "include"),
                        *defines, os.path.join(CSRC, "onebit_adam.cu")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout


def test_checks_compile_to_nothing_in_normal_builds():
    normal, checked = _preprocessed(), _preprocessed("-DONEBIT_CHECKS")
    for token in ("bounds_fail", "chunk_ok", "worker_unit_ok", "skip_bad_chunks", "A.check_margin"):
        assert token not in normal, token
        assert token in checked, token


def test_bounds_report_names_follow_the_kernel_enum():
    src = open(os.path.join(CSRC, "onebit_adam.cu")).read()
    m = re.search(r"names\[ONEBIT_NUM_KERNELS\]\s*=\s*\{([^}]*)\}", src)
    assert m, "the bounds report's kernel names"
    names = re.findall(r'"(\w+)"', m.group(1))
    assert names == ob.KERNEL_NAMES
