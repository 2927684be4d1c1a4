"""Benchmark of the 1-bit Adam compression-stage optimizer step on GB300.

A "step" is one compression-stage optimizer step over the whole synthetic parameter buffer with n
simulated workers: worker momentum + error feedback + 1-bit compression (worker kernel), worker
scales, server average + error feedback + recompression (server kernel), server scales, and the
preconditioned update.  Default workload: the BERT-Large-sized flat buffer (d = 340e6 fp32
parameters, n = 16 workers, fp16 gradients), warmed up with 20 uncompressed Adam steps before the
variance freeze.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl gb300|reference]

Under torchrun (N > 1) every rank runs an independent replica of the workload on its own GPU (its n
workers simulated inside that GPU); the timed region is bracketed by a barrier and a device
synchronisation and the slowest rank's time is reported.  With --exchange the n workers are instead
spread over the N GPUs (the multi-GPU form: an all-to-all and an all-gather of the compressed
messages per step).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HBM_NOMINAL_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def algorithmic_bytes(n: int, gb: int, step: str = "compress") -> dict:
    """Bytes per element each kernel must move in a steady-state step (compression stage: m carried
    as the broadcast's sign bits + one scale per shard; errors rebuilt from the stored c and a)."""
    if step == "warmup":
        k0 = n * gb + 24                        # n gradients; m, v, x read + write
        return {"warmup": k0, "step": k0}
    k2 = n / 8 + 4 + 4 + 1 / 8                  # n worker bit rows; a read + write; server bits
    if step == "ec_adam":
        k1 = n * (gb + 4 + 4 + 1 / 8)           # g_i, c_i read, c_i write, worker bits (no momentum)
        k3 = 1 / 8 + 8 + 8 + 8                  # server bits; m, v, x read + write
        return {"worker": k1, "server": k2, "ec_update": k3, "step": k1 + k2 + k3}
    k1 = n * (gb + 4 + 4 + 1 / 8) + 1 / 8      # g_i, c_i read, c_i write, worker bits; server bits
    k3 = 1 / 8 + 4 + 4 + 4                      # server bits; den; x read + write
    return {"worker": k1, "server": k2, "update": k3, "step": k1 + k2 + k3}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _kernel_source_hash(marker: str):
    """Hash of one kernel's source: the constants declared before it (the shared tuning constants
    and those of the kernels it builds on) plus the code of the kernel's own region (from its heading
    comment to the next separator), full-line comments left out."""
    import hashlib

    path = os.path.join(ROOT, "communication_compressed_optimizer_compress_gb300", "csrc", "onebit_kernels.cuh")
    src = open(path).read()
    i = src.index(marker)
    consts = "\n".join(ln for ln in src[:i].splitlines() if ln.startswith("constexpr "))
    j = src.index("\n// " + "-" * 40, i)  # the next full-width section separator
    code = "\n".join(ln for ln in src[i:j].splitlines() if not ln.lstrip().startswith("//"))  # comments aside
    return hashlib.sha256((consts + code).encode()).hexdigest()[:16]


def traffic_from_profiles(kernel: str, step: str, w, scale_block: int = 0):
    """DRAM bytes per launch of `kernel` in a `step` of workload `w`, from the committed ncu records
    (bytes per element there x the elements of this launch).  None when no record was taken on this
    shape (worker count, gradient width, number of tensors, scale block), when the kernel's source
    changed since the capture, or when the record does not scale to a full launch: at the capture's
    size the L2 absorbed more than 2% of the kernel's bytes (the previous kernel's output, or this
    kernel's last writes), and a share that large does not grow with the element count."""
    from communication_compressed_optimizer_compress_gb300 import workloads as W

    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            recs = json.load(f)
    except Exception:
        return None
    for rec in recs.values():
        if (rec["kernel"], rec["step"], rec["n_workers"], rec["grad_bytes"], rec["n_tensors"], rec["scale_block"]) != \
                (kernel, step, w.n_workers, W.GRAD_BYTES[w.grad_dtype], w.n_tensors, scale_block):
            continue
        if not rec["scales_to_launch"] or rec["source_sha256_16"] != _kernel_source_hash(rec["marker"]):
            return None
        return rec["dram_bytes_per_elem"] * w.d
    return None


def warmup_kernel(n: int, grad_bytes: int) -> str:
    """The warm-up kernel the library launches for aligned buffers: the staged variant for 16-bit
    gradients with kWarmStagedMin <= n <= kWarmStagedMax (constants read from the kernel source)."""
    path = os.path.join(ROOT, "communication_compressed_optimizer_compress_gb300", "csrc", "onebit_kernels.cuh")
    src = open(path).read()
    lo = int(re.search(r"constexpr int kWarmStagedMin = (\d+);", src).group(1))
    hi = int(re.search(r"constexpr int kWarmStagedMax = (\d+);", src).group(1))
    return "k_warmup_staged" if grad_bytes == 2 and lo <= n <= hi else "k_warmup"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------------- dist

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_max(value: float, device=None) -> float:
    """Maximum of a float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------------------- oracle

def host_cpu():
    """The host's core count and CPU model name (lscpu's "Model name", else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() == "Model name":
                model = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            for ln in open("/proc/cpuinfo"):
                if ln.lower().startswith(("model name", "cpu model")):
                    model = ln.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    return {"nproc": os.cpu_count(), "model": model}


class pinned_to_core0:
    """Run the enclosed host work on core 0 alone (the single-threaded oracle timing protocol)."""

    def __enter__(self):
        self.prev = None
        try:
            self.prev = os.sched_getaffinity(0)
            os.sched_setaffinity(0, {0})
            self.pinned = True
        except Exception:
            self.pinned = False
        return self

    def __exit__(self, *a):
        if self.prev is not None:
            try:
                os.sched_setaffinity(0, self.prev)
            except Exception:
                pass


def oracle_sample(w, seconds: float = 12.0, d_sample: int = 1 << 21):
    """Time the oracle (single-threaded C) on a bounded sample of the workload: the same worker
    count, gradient dtype and law on a flat buffer of d_sample parameters; one warm-up step, the
    freeze, then compression steps until `seconds` of wall time are spent.  Returns params/s."""
    import numpy as np

    import oracle
    from communication_compressed_optimizer_compress_gb300 import workloads as W

    ws = w.with_(numel=(d_sample,))
    src = W.GradSource(ws, "cpu")
    x0 = W.params(ws, "cpu")[0].numpy()
    o = oracle.OneBitAdamOracle([d_sample], ws.n_workers, x0, ws.beta1, ws.beta2, ws.eps, ws.lr,
                                grad_dtype=ws.grad_dtype)
    sets = [[W.to_numpy_grad(t) for t in src.grads(s)] for s in range(2)]
    o.warmup_step(sets[0])
    o.freeze()
    times = []
    with pinned_to_core0() as pin:
        t_all = time.perf_counter()
        k = 0
        while True:
            t0 = time.perf_counter()
            o.compress_step(sets[k % 2])
            times.append(time.perf_counter() - t0)
            k += 1
            if time.perf_counter() - t_all > seconds and k >= 1:
                break
    per = statistics.median(times)
    cpu = host_cpu()
    return {"value": d_sample / per, "unit": "params/s", "cores": 1, "kind": "oracle",
            "sample": f"{ws.name} law, flat d={d_sample} (a sample of the d={w.d} workload), n={ws.n_workers}, "
                      f"{W.DTYPE_NAME[ws.grad_dtype]} grads, {k} compression steps (median), single thread"
                      f"{' pinned to core 0' if pin.pinned else ''}",
            "d_sample": d_sample, "pinned_core0": pin.pinned, "host_nproc": cpu["nproc"], "host_cpu": cpu["model"],
            "s_per_step": per, "steps": k}


# ---------------------------------------------------------------------------------------- main

def run_reference(args, w):
    """The reference arm: the oracle (single-threaded C) on the host, W untimed then K timed
    compression steps, each on a bounded sample of the workload (the same worker count, gradient
    dtype and law on a flat buffer).  The sample starts at min(2^21, d) parameters and is halved
    (down to 2^15) until K steps take at most about a minute."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    from communication_compressed_optimizer_compress_gb300 import workloads as W

    budget_s = 60.0
    K, Wm = max(1, args.steps), max(1, args.warmup)

    def make(d):
        ws = w if d == w.d and args.ref_full else w.with_(numel=(d,))
        src = W.GradSource(ws, "cpu")
        o = oracle.OneBitAdamOracle([d], ws.n_workers, W.params(ws, "cpu")[0].numpy(), ws.beta1, ws.beta2, ws.eps,
                                    ws.lr, grad_dtype=ws.grad_dtype)
        sets = [[W.to_numpy_grad(t) for t in src.grads(s)] for s in range(2)]
        o.warmup_step(sets[0])
        o.freeze()
        return ws, o, sets

    if args.ref_full:  # the whole workload, no sample (minutes per step and tens of GB of host memory)
        d = w.d
        ws, o, sets = make(d)
        Wm = 0
    else:
        d = min(1 << 21, w.d)
        ws, o, sets = make(d)
        t0 = time.perf_counter()
        o.compress_step(sets[0])  # first warm-up step, also the size probe
        per = time.perf_counter() - t0
        while d > (1 << 15) and K * per * 1.1 > budget_s:
            d //= 2
            per /= 2
        if d != ws.d:
            ws, o, sets = make(d)
            o.compress_step(sets[0])
    with pinned_to_core0() as pin:
        for s in range(1, Wm):
            o.compress_step(sets[s % 2])
        t0 = time.perf_counter()
        for s in range(K):
            o.compress_step(sets[(Wm + s) % 2])
        total = time.perf_counter() - t0
    value = d * K / total
    ab = algorithmic_bytes(w.n_workers, W.GRAD_BYTES[w.grad_dtype])
    cpu = host_cpu()
    what = (f"{ws.name}, the whole workload ({ws.n_tensors} tensor(s), d={d})" if args.ref_full else
            f"{ws.name} law, flat d={d} (a sample of the d={w.d} workload)")
    sample = (f"{what}, n={ws.n_workers}, {W.DTYPE_NAME[ws.grad_dtype]} grads, {Wm} untimed + {K} timed "
              f"compression steps, single thread{' pinned to core 0' if pin.pinned else ''}")
    config = workload_config(w, args)
    config["d_sample"] = d  # the elements each timed oracle step processes; value = d_sample / step time
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": total / K * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config,
        "step_gbs": value * ab["step"] / 1e9,
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": 1, "kind": "oracle", "sample": sample,
                         "d_sample": d, "pinned_core0": pin.pinned, "host_nproc": cpu["nproc"],
                         "host_cpu": cpu["model"]},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_exchange(args, w):
    """The multi-GPU form: rank r of N simulates workers r*n/N .. (r+1)*n/N-1 and serves the same
    shards; a step is compress_begin, an all-to-all of the packed messages, compress_serve, an
    all-gather of the servers' results, compress_end.  value = d * steps / (slowest rank's time): the
    parameters one step updates, with the n workers' work spread over the N GPUs (strong scaling)."""
    import torch
    import torch.distributed as dist

    import communication_compressed_optimizer_compress_gb300 as ob
    from communication_compressed_optimizer_compress_gb300 import dist as D
    from communication_compressed_optimizer_compress_gb300 import workloads as W

    world, rank, local = dist_env()
    n = w.n_workers
    if args.emulate_ranks:
        return run_exchange_emulated(args, w, args.emulate_ranks)
    if n % world:
        raise SystemExit(f"--exchange needs the worker count ({n}) to be a multiple of the GPU count ({world})")
    nl, T = n // world, w.n_tensors
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    ob.lib()
    params = [p.to(dev) for p in W.params(w, dev)]
    src = W.GradSource(w, dev)
    gsets = []
    for s_ in range(2):  # this rank's workers' gradients only
        g = src.grads(s_)
        gsets.append(g[rank * nl * T:(rank + 1) * nl * T])
        del g
    opt = D.RankOneBitAdam(params, n, w.warmup_steps, rank, world,
                           transport=D.DeviceTransport() if world > 1 else D.LocalTransport(),
                           beta1=w.beta1, beta2=w.beta2, eps=w.eps, lr=w.lr, grad_dtype=W.TORCH_DTYPE[w.grad_dtype])
    stream = torch.cuda.current_stream()
    for s_ in range(w.warmup_steps):
        opt.warmup_step(gsets[s_ % 2])
    opt.freeze_variance()
    for s_ in range(max(3, args.warmup)):
        opt.compress_step(gsets[s_ % 2])
    torch.cuda.synchronize()
    assert opt.get_status() == ob.OK
    opt.set_timing(True)
    opt.kernel_times()
    launches0 = opt.launch_count()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        t0.record(stream)
        for s_ in range(args.steps):
            opt.compress_step(gsets[s_ % 2])
        t1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms = t0.elapsed_time(t1)
    max_ms = dist_max(ms, dev)
    kt = opt.kernel_times()
    launches = opt.launch_count() - launches0
    opt.set_timing(False)
    status = opt.get_status()
    gb = W.GRAD_BYTES[w.grad_dtype]
    ab_w = algorithmic_bytes(nl, gb)["worker"]           # this rank's workers, every element
    ab_s = algorithmic_bytes(n, gb)["server"] / world    # every worker's bits, this rank's shards
    ab_u = algorithmic_bytes(n, gb)["update"]            # the full replica
    ms_per_step = max_ms / args.steps
    wk_ms = kt["worker"][0] / max(1, kt["worker"][1])
    wk_gbs = w.d * ab_w / (wk_ms / 1e3) / 1e9 if wk_ms > 0 else None
    peak, peak_kind = measured_peak()
    per_kernel = {name: {"avg_ms": v[0] / max(1, v[1]), "launches": v[1]} for name, v in kt.items() if v[1]}
    if rank == 0:
        cfg = workload_config(w, args)
        cfg["parallelism"] = (f"multi-GPU form: {n} workers over {world} GPU(s) ({nl} per GPU); compressed "
                              f"all-to-all + all-gather ({'NCCL' if world > 1 else 'none at one GPU'})")
        line = {
            "metric": METRIC, "value": w.d * args.steps / (max_ms / 1e3), "unit": "params/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": cfg,
            "step_gbs_per_gpu": w.d * (ab_w + ab_s + ab_u) / (ms_per_step / 1e3) / 1e9,
            "exchange_bytes_per_step_per_gpu": opt.exchange_bytes(),
            "roofline": None if wk_gbs is None else {
                "bound": "hbm", "kernel": "k_worker (this GPU's workers)", "achieved": wk_gbs, "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": wk_gbs / peak, "traffic": None,
                "bytes_per_elem": ab_w, "elems_per_launch": w.d},
            "kernels": per_kernel, "gpu_launches": launches, "clocks": clk.summary(),
            "status": ob.error_string(status), "e2e": None, "cpu_baseline": None,
            "note": "one GPU: the split step with nothing to exchange" if world == 1 else None,
        }
        print(json.dumps(line), flush=True)
    opt.free()
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_exchange_emulated(args, w, R):
    """The multi-GPU form's per-rank work, measured on one GPU: R rank handles run one after another,
    the all-to-all and the all-gather replaced by the device copies they deliver.  Each rank's kernels
    (begin: its workers; serve: its shards; end: the update of its full replica) are timed with CUDA
    events; the copies standing in for the collectives are timed apart and are not a measure of any
    interconnect.  value = d * steps / (the slowest rank's kernel time): what R GPUs would reach if
    the exchange were free."""
    import torch

    import communication_compressed_optimizer_compress_gb300 as ob
    from communication_compressed_optimizer_compress_gb300 import dist as D
    from communication_compressed_optimizer_compress_gb300 import workloads as W

    n, T = w.n_workers, w.n_tensors
    if n % R:
        raise SystemExit(f"--emulate-ranks needs the worker count ({n}) to be a multiple of R ({R})")
    nl = n // R
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ob.lib()
    x0 = W.params(w, dev)
    src = W.GradSource(w, dev)
    gsets = [src.grads(s_) for s_ in range(2)]
    ranks = [D.RankOneBitAdam([t.clone() for t in x0], n, w.warmup_steps, r, R, transport=D.LocalTransport(),
                              beta1=w.beta1, beta2=w.beta2, eps=w.eps, lr=w.lr,
                              grad_dtype=W.TORCH_DTYPE[w.grad_dtype]) for r in range(R)]
    del x0
    stream = torch.cuda.current_stream()

    def step(s_, timed):
        g = gsets[s_ % 2]
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(3 * R + 2)] if timed else None
        k = 0

        def mark(i, fn):
            if timed:
                ev[i][0].record(stream)
            fn()
            if timed:
                ev[i][1].record(stream)
        for r, o in enumerate(ranks):
            mark(k, lambda: o.begin(g[r * nl * T:(r + 1) * nl * T])); k += 1
        if R > 1:
            mark(k, lambda: [o.recv.view(R, -1).copy_(torch.stack([ranks[p].send.view(R, -1)[q] for p in range(R)]))
                             for q, o in enumerate(ranks)])
        k += 1
        for o in ranks:
            mark(k, o.serve); k += 1
        if R > 1:
            cat = torch.cat([o.bcast for o in ranks])
            mark(k, lambda: [o.gathered.copy_(cat) for o in ranks])
        k += 1
        for o in ranks:
            mark(k, o.end); k += 1
        return ev

    for s_ in range(w.warmup_steps):
        for o in ranks:
            ob.OneBitAdam.warmup_step(o, gsets[s_ % 2])
    for o in ranks:
        o.freeze_variance()
    for s_ in range(max(3, args.warmup)):
        step(s_, False)
    torch.cuda.synchronize()
    per_rank = [0.0] * R
    copies = 0.0
    records = [step(s_, True) for s_ in range(args.steps)]
    torch.cuda.synchronize()
    for ev in records:
        el = [a.elapsed_time(b) if R > 1 or i not in (R, 2 * R + 1) else 0.0 for i, (a, b) in enumerate(ev)]
        for r in range(R):
            per_rank[r] += el[r] + el[R + 1 + r] + el[2 * R + 2 + r]
        copies += el[R] + el[2 * R + 1]
    per_rank = [v / args.steps for v in per_rank]
    status = max(o.get_status() for o in ranks)
    line = {
        "metric": METRIC + " (multi-GPU form, per-rank kernels emulated on one GPU)",
        "value": w.d / (max(per_rank) / 1e3), "unit": "params/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max(per_rank), "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(workload_config(w, args), parallelism=f"{R} emulated ranks x {nl} workers"),
        "emulated_ranks": R, "per_rank_kernel_ms": per_rank,
        "collective_stand_in_copies_ms_per_step": copies / args.steps,
        "exchange_bytes_per_step_per_rank": ranks[0].exchange_bytes(),
        "status": ob.error_string(status),
        "note": "each rank's kernels measured on this GPU one rank at a time; the interconnect time is not "
                "measured: value and ms_per_step assume the exchange is free",
    }
    print(json.dumps(line), flush=True)
    for o in ranks:
        o.free()
    return 0


METRIC = "compression-stage optimizer step params/s and HBM GB/s (% of 8 TB/s) at 1 GB300"
STEP_METRIC = {
    "warmup": "warm-up (uncompressed) Adam step params/s and HBM GB/s at 1 GB300",
    "ec_adam": "gradient-compression baseline step (1-bit EC on gradients + Adam) params/s and HBM GB/s at 1 GB300",
}


def workload_config(w, args):
    from communication_compressed_optimizer_compress_gb300 import workloads as W

    desc = (f"{w.name}: {w.n_tensors} tensor(s), d={w.d} fp32 params, n={w.n_workers} simulated workers, "
            f"{W.DTYPE_NAME[w.grad_dtype]} grads ({w.law}), T_w={w.warmup_steps} Adam steps then timed "
            f"compression steps")
    return {"workload": desc, "d": w.d, "n_tensors": w.n_tensors, "n_workers": w.n_workers,
            "grad_dtype": W.DTYPE_NAME[w.grad_dtype], "warmup_adam_steps": w.warmup_steps,
            "l2": "inputs larger than L2 (working set per step >> 129 MB); no flush needed",
            "parallelism": f"replicas x{dist_env()[0]} (workers simulated in one GPU)",
            "scale_block": getattr(args, "scale_block", 0)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="bert_large")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--d", type=int, default=0, help="override the parameter count (flat workloads)")
    ap.add_argument("--tw", type=int, default=-1, help="override the number of warm-up Adam steps")
    ap.add_argument("--n", type=int, default=0, help="override the number of simulated workers")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--step", default="compress", choices=["compress", "warmup", "ec_adam"],
                    help="what one timed step is: the compression-stage step (default), an uncompressed "
                         "warm-up Adam step, or the gradient-compression baseline step")
    ap.add_argument("--graph", action="store_true",
                    help="capture two steps (one cycle of the double-buffered scales) in a CUDA graph and "
                         "time its replays; per-kernel events are off, so no roofline is reported")
    ap.add_argument("--scale-block", type=int, default=0,
                    help="per-block scale granularity: every block of this many elements (a multiple of 32) "
                         "gets its own worker scales and server shards; 0 = per tensor")
    ap.add_argument("--ref-full", action="store_true",
                    help="with --impl reference: time the oracle on the whole workload instead of a sample")
    ap.add_argument("--emulate-ranks", type=int, default=0,
                    help="with --exchange at one GPU: run R ranks' handles one after another on this GPU, the "
                         "collectives replaced by the device copies they deliver, and report each rank's kernel "
                         "time (the interconnect is not measured)")
    ap.add_argument("--exchange", action="store_true",
                    help="the multi-GPU form: the n workers split over the ranks (n/N per GPU), the compressed "
                         "messages exchanged with an NCCL all-to-all and all-gather between the library's split "
                         "step calls; at one GPU the split step with nothing to exchange")
    args = ap.parse_args()
    if args.graph and args.steps % 2:
        args.steps += 1

    from communication_compressed_optimizer_compress_gb300 import workloads as W

    w = W.WORKLOADS[args.config]
    if args.d:
        w = w.with_(numel=(args.d,))
    if args.tw >= 0:
        w = w.with_(warmup_steps=max(1, args.tw))
    if args.n > 0:
        w = w.with_(n_workers=args.n)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.exchange:
        return run_exchange(args, w)

    import torch
    import torch.distributed as dist

    import communication_compressed_optimizer_compress_gb300 as ob

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    ob.lib()  # fail loudly if the library is missing

    # ---- inputs resident in HBM: parameters, two gradient sets alternated between steps
    params = [p.to(dev) for p in W.params(w, dev)]
    src = W.GradSource(w, dev)
    gsets = [src.grads(s) for s in range(2)]
    # a timed warm-up step needs room for the untimed and timed warm-up steps before T_w
    tw_handle = w.warmup_steps if args.step == "compress" else args.warmup + args.steps + 1
    opt = ob.OneBitAdam(params, w.n_workers, tw_handle, w.beta1, w.beta2, w.eps, w.lr,
                        grad_dtype=W.TORCH_DTYPE[w.grad_dtype], scale_block=args.scale_block)
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    warm_ms = None
    if args.step == "compress":
        t0.record(stream)
        for s in range(w.warmup_steps):
            opt.warmup_step(gsets[s % 2])
        t1.record(stream)
        torch.cuda.synchronize()
        warm_ms = t0.elapsed_time(t1) / max(1, w.warmup_steps)
        opt.freeze_variance()
        step_fn = opt.compress_step
    elif args.step == "warmup":
        step_fn = opt.warmup_step
    else:
        step_fn = opt.ec_adam_step
    first_ms = None
    for s in range(max(3, args.warmup)):
        if s == 0 and args.step == "compress":  # the first step after the freeze reads the fp32 m
            t0.record(stream)
            step_fn(gsets[0])
            t1.record(stream)
            torch.cuda.synchronize()
            first_ms = t0.elapsed_time(t1)
            continue
        step_fn(gsets[s % 2])
    assert opt.get_status() == ob.OK, "non-finite state after warm-up"

    # ---- optional CUDA graph of two steps (the gradient-pointer tables are cached by the steps above)
    graph = None
    if args.graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        c0 = opt.launch_count()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                step_fn(gsets[0])
                step_fn(gsets[1])
        stream.wait_stream(side)
        launches_per_replay = opt.launch_count() - c0
        graph.replay()
        torch.cuda.synchronize()

    # ---- timed region
    opt.set_timing(graph is None)
    opt.kernel_times()  # reset
    launches0 = opt.launch_count()
    barrier()
    torch.cuda.synchronize()
    n_marks = args.steps if graph is None else args.steps // 2
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(n_marks)]
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        t0.record(stream)
        if graph is None:
            for s in range(args.steps):
                step_fn(gsets[s % 2])
                marks[s].record(stream)
        else:
            for r in range(args.steps // 2):
                graph.replay()
                marks[r].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    barrier()
    elapsed_ms = t0.elapsed_time(t1)
    per_mark = args.steps / n_marks
    step_times = sorted([t0.elapsed_time(marks[0]) / per_mark] +
                        [marks[i - 1].elapsed_time(marks[i]) / per_mark for i in range(1, n_marks)])

    def pct(q):
        return step_times[min(len(step_times) - 1, int(q * (len(step_times) - 1) + 0.5))]
    if graph is None:
        launches = opt.launch_count() - launches0
        kt = opt.kernel_times()
    else:
        launches = launches_per_replay * (args.steps // 2)
        kt = {name: (0.0, 0) for name in opt.kernel_times()}
    opt.set_timing(False)
    max_ms = dist_max(elapsed_ms, dev)
    status = opt.get_status()

    ab = algorithmic_bytes(w.n_workers, W.GRAD_BYTES[w.grad_dtype], args.step)
    ms_per_step = max_ms / args.steps
    value = world * w.d * args.steps / (max_ms / 1e3)
    step_gbs = w.d * ab["step"] / (ms_per_step / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    dom = "warmup" if args.step == "warmup" else "worker"
    warm_kernel = warmup_kernel(w.n_workers, W.GRAD_BYTES[w.grad_dtype])
    # the kernel behind each timing bucket (the server's staged variant on the shapes it has records for)
    bucket_kernel = {"warmup": warm_kernel, "worker": "k_worker", "server": "k_server_staged", "update": "k_update",
                     "ec_update": "k_ec_adam_update"}
    dom_ms = kt[dom][0] / max(1, kt[dom][1])
    dom_gbs = w.d * ab[dom] / (dom_ms / 1e3) / 1e9 if dom_ms > 0 else None
    per_kernel = {}
    for name in ("warmup", "worker", "worker_scale", "server", "server_scale", "update", "ec_update"):
        ms, cnt = kt[name]
        if not cnt:
            continue
        avg = ms / max(1, cnt)
        entry = {"avg_ms": avg, "launches": cnt, "share": ms / max(1e-9, sum(v[0] for v in kt.values()))}
        if name in ab:
            entry["gbs"] = w.d * ab[name] / (avg / 1e3) / 1e9
            entry["bytes_per_elem"] = ab[name]
        if name in bucket_kernel:
            entry["traffic"] = traffic_from_profiles(bucket_kernel[name], args.step, w, args.scale_block)
        per_kernel[name] = entry

    # ---- end to end through the C ABI with host gradient buffers (H2D copies inside the timing)
    e2e = None
    if not args.no_e2e and args.step == "compress":
        host = []
        for g in gsets[0]:
            hb = torch.empty(g.shape, dtype=g.dtype, pin_memory=True)
            hb.copy_(g)
            host.append(hb)
        h2d = sum(t.numel() * t.element_size() for t in host)
        out = torch.empty(w.n_tensors * w.n_workers, dtype=torch.float32).pin_memory()
        e2e_steps = max(2, min(args.steps, 10))
        opt.compress_step_host(host)  # first call allocates the library's staging buffer
        torch.cuda.synchronize()

        probe_streams = [torch.cuda.Stream(device=dev) for _ in range(4)]

        def link_probe():
            """The host link at this moment: plain copies of this step's own host gradients into
            device buffers of the same shapes, cut the way the library cuts its staging copies
            (64 MB pieces, round-robin over 4 streams) with nothing else running, in GB/s."""
            t0.record(stream)
            for cs in probe_streams:
                cs.wait_stream(stream)
            r = 0
            for hb, db in zip(host, gsets[1]):
                src, dst = hb.view(-1), db.view(-1)
                piece = (64 << 20) // hb.element_size()
                for a in range(0, src.numel(), piece):
                    with torch.cuda.stream(probe_streams[r % 4]):
                        dst[a:a + piece].copy_(src[a:a + piece], non_blocking=True)
                    r += 1
            for cs in probe_streams:
                stream.wait_stream(cs)
            t1.record(stream)
            torch.cuda.synchronize()
            return h2d / (t0.elapsed_time(t1) / 1e3) / 1e9

        link_before = link_probe()
        barrier()
        t0.record(stream)
        for s in range(e2e_steps):
            opt.compress_step_host(host)
            out.copy_(opt.export_state(ob.STATE_SERVER_SCALES), non_blocking=True)
        t1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = dist_max(t0.elapsed_time(t1), dev)
        link_after = link_probe()
        link_gbs = max(link_before, link_after)
        moved = h2d / (e2e_ms / e2e_steps / 1e3) / 1e9
        e2e = {"value": world * w.d * e2e_steps / (e2e_ms / 1e3), "unit": "params/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": out.numel() * 4,
               "ms_per_step": e2e_ms / e2e_steps,
               "link_h2d_gbs": link_gbs,
               "link_h2d_gbs_before_after": [link_before, link_after],
               "frac_of_link": moved / link_gbs,
               "frac_of_link_before_after": [moved / link_before, moved / link_after],
               "params_on_device": True,
               "path": "onebit_adam_compress_step_host (pinned host grads copied in by the library) + D2H of "
                       "the server scales; the updated parameters and the optimizer state stay in HBM, as in a "
                       "training loop, so only the scales come back"}
        del host

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.step == "compress":
        cb = oracle_sample(w)
        cpu = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample", "d_sample", "pinned_core0", "host_nproc",
                                  "host_cpu")}

    if rank == 0:
        line = {
            "metric": METRIC if args.step == "compress" else STEP_METRIC[args.step], "value": value, "unit": "params/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(w, args),
            "step_gbs": step_gbs, "step_pct_of_8tbs": 100.0 * step_gbs / HBM_NOMINAL_GBS,
            "step_frac_of_measured_peak": step_gbs / peak,
            "bytes_per_elem": ab["step"],
            "roofline": None if dom_gbs is None else {"bound": "hbm",
                         "kernel": {"compress": "k_worker (momentum + error + sign pack + norm partials)",
                                    "ec_adam": "k_worker (gradient + error + sign pack + norm partials)",
                                    "warmup": f"{warm_kernel} (worker mean + Adam)"}[args.step],
                         "achieved": dom_gbs, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": dom_gbs / peak,
                         "traffic": traffic_from_profiles(bucket_kernel[dom], args.step, w, args.scale_block),
                         "bytes_per_elem": ab[dom], "elems_per_launch": w.d},
            "kernels": per_kernel,
            "warmup_adam_ms_per_step": warm_ms,
            "step_ms_p10_p50_p90": [pct(0.1), pct(0.5), pct(0.9)],
            "first_compress_step_ms": first_ms,
            "gpu_launches": launches,
            "cuda_graph": graph is not None,
            "clocks": clk.summary(),
            "status": ob.error_string(status),
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    opt.free()
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
