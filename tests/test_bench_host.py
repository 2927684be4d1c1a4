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
    keys = set()
    for name, rec in _records().items():
        for key in ("kernel", "step", "n_workers", "grad_bytes", "n_tensors", "scale_block", "dram_bytes_per_elem",
                    "scales_to_launch", "marker", "source_sha256_16", "captured_on", "summary"):
            assert key in rec, (name, key)
        shape = (rec["kernel"], rec["step"], rec["n_workers"], rec["grad_bytes"], rec["n_tensors"], rec["scale_block"])
        assert shape not in keys, name  # one record per kernel, step and shape
        keys.add(shape)
        assert os.path.isfile(os.path.join(ROOT, rec["summary"])), rec["summary"]
        assert rec["step"] in ("compress", "warmup", "ec_adam")
        # traffic is a measurement of the algorithmic bytes: never far above, a little below when
        # the previous kernel's output (or this one's last writes) are still in L2
        alg = bench.algorithmic_bytes(rec["n_workers"], rec["grad_bytes"], rec["step"])
        bucket = {"k_worker": "worker", "k_server_staged": "server", "k_warmup_staged": "warmup", "k_warmup": "warmup",
                  "k_update": "update", "k_ec_adam_update": "ec_update"}[rec["kernel"]]
        assert 0.75 * alg[bucket] <= rec["dram_bytes_per_elem"] <= 1.05 * alg[bucket], (name, alg[bucket])
        # only a record whose capture lost at most 2% to L2 is scaled to a full launch
        assert rec["scales_to_launch"] == (rec["dram_bytes_per_elem"] >= 0.98 * alg[bucket]), name


def test_traffic_lookup_matches_workload_and_source(monkeypatch):
    from communication_compressed_optimizer_compress_gb300 import workloads as W

    w = W.WORKLOADS["bert_large"]
    rec = next(r for r in _records().values() if r["kernel"] == "k_worker" and r["step"] == "compress")
    assert (rec["n_workers"], rec["grad_bytes"], rec["n_tensors"]) == (w.n_workers, W.GRAD_BYTES[w.grad_dtype], 1)
    live = bench._kernel_source_hash(rec["marker"]) == rec["source_sha256_16"]
    got = bench.traffic_from_profiles("k_worker", "compress", w)
    assert got == (rec["dram_bytes_per_elem"] * w.d if live else None)
    # another shape has no record: null, never the figure of a different configuration
    assert bench.traffic_from_profiles("k_worker", "compress", w.with_(n_workers=8)) is None
    assert bench.traffic_from_profiles("k_worker", "compress", w.with_(grad_dtype=W.F32)) is None
    assert bench.traffic_from_profiles("k_worker", "compress", w.with_(numel=(1000, 2000))) is None
    assert bench.traffic_from_profiles("k_worker", "compress", w, scale_block=65536) is None
    assert bench.traffic_from_profiles("k_worker", "warmup", w) is None
    assert bench.traffic_from_profiles("no_such_kernel", "compress", w) is None
    # a record that does not scale to a full launch is never scaled
    for rec in _records().values():
        if not rec["scales_to_launch"]:
            shape = w.with_(n_workers=rec["n_workers"], grad_dtype={2: W.F16, 4: W.F32}[rec["grad_bytes"]])
            assert bench.traffic_from_profiles(rec["kernel"], rec["step"], shape) is None, rec["kernel"]
    # a kernel whose source changed since the capture reads as null
    monkeypatch.setattr(bench, "_kernel_source_hash", lambda marker: "0" * 16)
    assert bench.traffic_from_profiles("k_worker", "compress", w) is None


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
