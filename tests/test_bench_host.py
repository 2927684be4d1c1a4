"""Host-side logic of bench.py: the committed DRAM-traffic records, their lookup, the algorithmic
byte counts behind every roofline figure, and the warm-up kernel label.  No GPU needed."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _records():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        return json.load(f)


def test_traffic_records_are_complete():
    for name, rec in _records().items():
        for key in ("dram_bytes_per_elem", "n_workers", "grad_bytes", "step", "marker", "source_sha256_16",
                    "captured_on", "summary"):
            assert key in rec, (name, key)
        assert os.path.isfile(os.path.join(ROOT, rec["summary"])), rec["summary"]
        assert rec["step"] in ("compress", "warmup", "ec_adam")
        # traffic is a measurement of the algorithmic bytes: never far above, a little below when
        # the previous kernel's output is still in L2
        alg = bench.algorithmic_bytes(rec["n_workers"], rec["grad_bytes"], rec["step"])
        key = {"k_worker": "worker", "k_worker[ec_adam]": "worker", "k_server_staged": "server",
               "k_warmup_staged": "warmup"}[name]
        assert 0.75 * alg[key] <= rec["dram_bytes_per_elem"] <= 1.05 * alg[key], (name, alg[key])


def test_traffic_lookup_matches_workload_and_source(monkeypatch):
    recs = _records()
    rec = recs["k_worker"]
    d = 340_000_000
    live = bench._kernel_source_hash(rec["marker"]) == rec["source_sha256_16"]
    got = bench.traffic_from_profiles("k_worker", rec["n_workers"], rec["grad_bytes"], d)
    assert got == (rec["dram_bytes_per_elem"] * d if live else None)
    # another worker count or gradient width has no record: null, never the n=16 figure
    assert bench.traffic_from_profiles("k_worker", rec["n_workers"] // 2, rec["grad_bytes"], d) is None
    assert bench.traffic_from_profiles("k_worker", rec["n_workers"], 4, d) is None
    assert bench.traffic_from_profiles("no_such_kernel", 16, 2, d) is None
    # a kernel whose source changed since the capture reads as null
    monkeypatch.setattr(bench, "_kernel_source_hash", lambda marker: "0" * 16)
    assert bench.traffic_from_profiles("k_worker", rec["n_workers"], rec["grad_bytes"], d) is None


def test_algorithmic_bytes_closed_forms():
    """B = n(gb + 8.25) + 20.375 for the compression step; n·gb + 24 for a warm-up step."""
    for n in (1, 2, 4, 8, 16, 33, 256):
        for gb in (2, 4):
            c = bench.algorithmic_bytes(n, gb, "compress")
            assert c["step"] == pytest.approx(n * (gb + 8.25) + 20.375)
            assert c["worker"] + c["server"] + c["update"] == pytest.approx(c["step"])
            wm = bench.algorithmic_bytes(n, gb, "warmup")
            assert wm["step"] == wm["warmup"] == n * gb + 24
            e = bench.algorithmic_bytes(n, gb, "ec_adam")
            assert e["step"] == pytest.approx(e["worker"] + e["server"] + e["ec_update"])
    assert bench.algorithmic_bytes(16, 2)["step"] == pytest.approx(184.375)


def test_warmup_kernel_label_follows_the_dispatch_rule():
    assert bench.warmup_kernel(16, 2) == "k_warmup_staged"
    assert bench.warmup_kernel(8, 2) == "k_warmup_staged"
    assert bench.warmup_kernel(20, 2) == "k_warmup_staged"
    assert bench.warmup_kernel(7, 2) == "k_warmup"
    assert bench.warmup_kernel(21, 2) == "k_warmup"
    assert bench.warmup_kernel(16, 4) == "k_warmup"
