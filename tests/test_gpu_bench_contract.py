"""The benchmark's JSON line, as the runs that consume it expect it: every key, with the right kinds
of values, for the compression step (with the roofline, end-to-end and CPU-baseline legs) and for
the reference arm."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_bench_line_has_every_key():
    d = _run("--config", "tiny", "--steps", "4", "--warmup", "3")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks", "cpu_baseline"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 4 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["data"] == "synthetic" and d["value"] > 0 and d["ms_per_step"] > 0
    assert "workload" in d["config"]
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    e = d["e2e"]
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in e, k
    assert e["unit"] == d["unit"] and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    c = d["clocks"]
    for k in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert k in c, k
    b = d["cpu_baseline"]
    for k in ("value", "unit", "cores", "kind", "sample", "d_sample", "host_nproc", "host_cpu", "pinned_core0"):
        assert k in b, k
    assert b["kind"] == "oracle" and b["cores"] >= 1
    assert d["gpu_launches"] == 6 * 4  # six kernels per compression step


def test_reference_arm_line():
    d = _run("--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1")
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert 0 < d["config"]["d_sample"] <= d["config"]["d"]  # the timed sample is stated beside the workload
