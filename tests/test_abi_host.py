"""The C-ABI library without a GPU: it loads, exports every declared symbol, validates configs and
plans its chunk table (the multi-tensor launcher) correctly.  No compute call is made here."""
import ctypes
import os
import re

import numpy as np
import pytest

import communication_compressed_optimizer_compress_gb300 as ob
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from communication_compressed_optimizer_compress_gb300 import _build

    _build.build()


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(onebit_\w+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert len(names) >= 20, names
    L = ctypes.CDLL(ob.LIB_PATH)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_error_strings():
    for s in range(9):
        assert ob.error_string(s) and "unknown" not in ob.error_string(s)
    assert "unknown" in ob.error_string(99)


@pytest.mark.parametrize("kw,bad", [
    (dict(numel=[0]), "empty"), (dict(numel=[-1, 5]), "negative"), (dict(n_workers=0), "n=0"),
    (dict(n_workers=257), "n too large"), (dict(beta1=1.0), "beta1"), (dict(beta2=-0.1), "beta2"),
    (dict(eps=-1.0), "eps"), (dict(warmup_steps=0), "T_w"), (dict(grad_dtype=3), "dtype"),
    (dict(scale_block=-32), "negative block"), (dict(scale_block=48), "block not a multiple of 32"),
])
def test_config_validation(kw, bad):
    base = dict(numel=[100], n_workers=2, warmup_steps=1)
    base.update(kw)
    cfg = ob.make_config(**base)
    with pytest.raises(ob.OneBitError) as e:
        ob.workspace_size(cfg)
    assert e.value.status == ob.ERR_INVALID_ARG


def test_null_arguments_return_status():
    L = ob.lib()
    assert L.onebit_adam_workspace_size(None, None) == ob.ERR_INVALID_ARG
    assert L.onebit_adam_free(None) == ob.ERR_INVALID_ARG
    assert L.onebit_adam_compress_step(None, None, None) == ob.ERR_INVALID_ARG
    assert L.onebit_adam_get_status(None, None) == ob.ERR_INVALID_ARG
    cfg = ob.make_config([10], 2)
    assert L.onebit_adam_init(ctypes.byref(cfg), None, None, 0, None, None) == ob.ERR_INVALID_ARG


SHAPES = [[1], [5, 0, 33, 200], [65536 * 3 + 17], [1 << 20], [1000] * 7, [110_000_000], [1, 1, 1]]


def _check_server_plan(numel, n, block=0):
    """Server-side chunks tile every segment (a tensor, or a scale block of one) exactly once, never
    cross a server shard (the oracle's shard rule), start on a 32-element boundary, hold at most
    65536 elements, and keep the caller's padded element offsets."""
    segs = oracle.scale_blocks(numel, block)
    rows = ob.plan_chunks(ob.make_config(numel, n, scale_block=block))
    by_seg = {k: [] for k in range(len(segs))}
    for (k, j, start, length, off) in rows:
        by_seg[k].append((j, start, length, off))
        assert 1 <= length <= 65536 and start % 32 == 0 and off % 32 == 0
    pad_starts, pad_off = [], 0
    for L in numel:
        pad_starts.extend(pad_off + s for s in (range(0, L, block) if (L and block) else [0]))
        pad_off += (L + 31) // 32 * 32
    assert len(pad_starts) == len(segs)
    for k, L in enumerate(segs):
        pos = 0
        for (j, start, length, off) in by_seg[k]:
            assert start == pos
            lo, hi = oracle.shard(L, n, j)
            assert lo <= start and start + length <= hi
            assert off == pad_starts[k] + start
            pos += length
        assert pos == L
    return rows


def _check_worker_plan(numel, n, block=0):
    """Worker chunks tile every segment once, start on a 32-element boundary, hold at most one chunk
    length; a chunk that spans shards holds whole shards (its first shard and the recorded shard
    length follow the oracle's shard rule); where shards are at least a chunk long the worker table
    equals the server-side table."""
    cfg = ob.make_config(numel, n, scale_block=block)
    rows = ob.plan_worker_chunks(cfg)
    server = ob.plan_chunks(cfg)
    segs = oracle.scale_blocks(numel, block)
    want = -(-sum(numel) // 1216)
    clen = min(65536, max(4096, -(-want // 4096) * 4096))  # the chunk-length rule
    by_seg = {k: [] for k in range(len(segs))}
    for r in rows:
        by_seg[r[0]].append(r)
    for k, L in enumerate(segs):
        per = 32 * -(-L // (32 * n)) if L else 0
        pos = 0
        for (seg, j, start, length, off, rper) in by_seg[k]:
            assert start == pos and start % 32 == 0 and 1 <= length <= 65536
            lo, hi = oracle.shard(L, n, j)
            assert lo == start if rper else lo <= start < hi
            if rper:
                assert rper == per and start % per == 0 and length > per
                last = (start + length - 1) // per
                assert last < n and (start + length == L or (start + length) % per == 0)
            else:
                assert start + length <= hi
            pos += length
        assert pos == L
        if per >= clen:
            assert [r[:5] for r in by_seg[k]] == [r for r in server if r[0] == k]
    return rows


@pytest.mark.parametrize("numel", SHAPES, ids=lambda v: f"T{len(v)}_{sum(v)}")
@pytest.mark.parametrize("n", [1, 3, 8, 16])
def test_chunk_plan(numel, n):
    """The server-side table on fixed shapes (see _check_server_plan)."""
    _check_server_plan(numel, n)


def _random_plan_configs(count, seed):
    """Seeded random lists: empty, tiny, ragged and multi-chunk tensors, worker counts 1..256, and
    per-tensor or per-block scales."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        T = int(rng.integers(1, 41))
        kind = rng.choice(5, size=T, p=[0.05, 0.2, 0.35, 0.35, 0.05])
        lo = np.array([0, 1, 65, 5000, 1_000_000])[kind]
        hi = np.array([1, 65, 5000, 300_000, 3_000_000])[kind]
        numel = [int(rng.integers(a, b)) for a, b in zip(lo, hi)]
        if not sum(numel):  # a list with no element at all is refused by design
            numel[-1] = 1
        n = int(rng.choice([1, 2, 3, 5, 7, 8, 13, 16, 17, 31, 64, 128, 200, 256]))
        block = 0 if rng.random() < 0.6 else 32 * int(rng.integers(1, 4097))
        out.append((numel, n, block))
    return out


@pytest.mark.parametrize("numel,n,block", _random_plan_configs(200, 2024),
                         ids=lambda v: None if not isinstance(v, list) else f"T{len(v)}")
def test_random_plans(numel, n, block):
    """Both tables on seeded random configurations, against the oracle's shard and blocking rules."""
    _check_server_plan(numel, n, block)
    _check_worker_plan(numel, n, block)


@pytest.mark.parametrize("numel,n,block", [([224, 0, 96], 2, 64), ([5000, 37], 20, 32), ([1 << 20], 4, 4096),
                                            ([65536 * 3 + 17, 5], 3, 96), ([100], 4, 1 << 20)])
def test_chunk_plan_scale_blocks(numel, n, block):
    """With a scale block, the plan's segments are the blocks of the oracle's blocking rule (blocks
    are multiples of 32, so only a tensor's last block can be ragged); see _check_server_plan."""
    _check_server_plan(numel, n, block)


WORKER_PLANS = [([1 << 20], 4, 0), ([1000], 16, 0), ([5, 0, 33, 200], 4, 0), ([340_000_000], 16, 0),
                ([224, 0, 96], 3, 96), ([1 << 20], 16, 65536), ([70_001, 33, 0, 5], 3, 96), ([5000], 20, 32)]


@pytest.mark.parametrize("numel,n,block", WORKER_PLANS, ids=[f"{sum(a)}_n{b}_B{c}" for a, b, c in WORKER_PLANS])
def test_worker_chunk_plan(numel, n, block):
    """The worker table on fixed shapes (see _check_worker_plan)."""
    _check_worker_plan(numel, n, block)


def test_oversized_plans_are_refused_before_they_are_built():
    """A tiny scale block on a huge tensor (2^40 elements in blocks of 32), a list too long for
    32-bit segment indices, or more than 2^40 elements in all is ONEBIT_ERR_UNSUPPORTED, returned at
    once, without building the plan."""
    import time

    for numel, n, block in (([1 << 40], 16, 32), ([1 << 36], 256, 32), ([1 << 40, 1], 2, 0), ([1 << 41], 1, 0)):
        t = time.perf_counter()
        with pytest.raises(ob.OneBitError) as e:
            ob.workspace_size(ob.make_config(numel, n, scale_block=block))
        assert e.value.status == ob.ERR_UNSUPPORTED
        assert time.perf_counter() - t < 1.0


def test_small_lists_get_short_chunks():
    """Chunk length adapts to the list: 2^20 elements become 256 chunks of 4096 (work units for
    every SM), while a BERT-Large-sized list keeps 65536-element chunks."""
    rows = ob.plan_chunks(ob.make_config([1 << 20], 1))
    assert len(rows) == 256 and all(r[3] == 4096 for r in rows)
    rows = ob.plan_chunks(ob.make_config([340_000_000], 16))
    assert max(r[3] for r in rows) == 65536


def test_workspace_size_scales_with_workers():
    a = ob.workspace_size(ob.make_config([1 << 20], 2))
    b = ob.workspace_size(ob.make_config([1 << 20], 4))
    # two more workers: two compensated-momentum rows (4 B/elem) and two sign rows (1/8 B/elem)
    assert b - a >= 2 * (1 << 20) * 4 + 2 * (1 << 20) // 8


def test_comm_bytes_volume_reduction_closed_form():
    """The message of one worker is ceil(L/32) words + one scale per tensor: 1/32 of fp32."""
    numel = [340_000_000]
    compressed = sum(((L + 31) // 32) * 4 + 4 for L in numel)
    assert abs(compressed / (4 * numel[0]) - 1 / 32) < 1e-6


def test_missing_library_raises_instead_of_falling_back(monkeypatch):
    """Without the built library every entry point raises at once: there is no CPU path."""
    pkg = ob
    monkeypatch.setattr(pkg, "_lib", None)
    monkeypatch.setattr(pkg, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libonebit_adam.so"))
    with pytest.raises(RuntimeError, match="missing"):
        pkg.lib()
    with pytest.raises(RuntimeError, match="missing"):
        pkg.workspace_size(pkg.make_config([10], 2))


def test_binding_refuses_host_or_non_fp32_parameters():
    """The optimizer takes contiguous fp32 CUDA tensors only; anything else is refused before the
    library is called."""
    import torch

    for bad in (torch.zeros(64), torch.zeros(64, dtype=torch.float64), torch.zeros(8, 8).t()):
        with pytest.raises(ValueError, match="fp32 CUDA"):
            ob.OneBitAdam([bad], 2, 1)


def test_failed_init_keeps_its_message_without_a_handle():
    """On a host with no CUDA device, init fails with ONEBIT_ERR_CUDA, returns no handle, and the
    CUDA message is available from onebit_adam_last_error(NULL) (a failed init has no handle)."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("needs a host without a CUDA device")
    L = ob.lib()
    cfg = ob.make_config([1024], 2)
    ptrs = (ctypes.c_void_p * 1)(0x1000)  # never dereferenced: there is no device to reach
    h = ctypes.c_void_p()
    assert L.onebit_adam_init(ctypes.byref(cfg), ptrs, None, 0, None, ctypes.byref(h)) == ob.ERR_CUDA
    assert not h.value
    assert "cudaGetDevice" in L.onebit_adam_last_error(None).decode()
    with pytest.raises(ob.OneBitError, match="cudaGetDevice"):
        ob._check(ob.ERR_CUDA, "onebit_adam_init")


def test_header_is_plain_c(tmp_path):
    """include/onebit_adam.h is a C header: it compiles as C99 and as C++ with no CUDA or torch
    header, and a C program can take the address of every entry point it declares."""
    import shutil
    import subprocess

    hdr = os.path.join(ROOT, "include", "onebit_adam.h")
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(onebit_\w+)\(", open(hdr).read(), re.M)
    assert len(names) >= 20
    src = tmp_path / "use.c"
    src.write_text('#include "onebit_adam.h"\n'
                   "typedef void (*entry_t)(void);\n"
                   "entry_t table[] = {\n" + ",\n".join(f"  (entry_t){n}" for n in names) + "\n};\n")
    for cc, std in (("gcc", "-std=c99"), ("g++", "-std=c++17")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not available")
        lang = ["-x", "c++"] if cc == "g++" else []
        r = subprocess.run([cc, *lang, std, "-Wall", "-Werror", "-pedantic", "-fsyntax-only",
                            "-I", os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def _kernel_constant(name):
    src = open(os.path.join(ROOT, "communication_compressed_optimizer_compress_gb300", "csrc", "onebit_kernels.cuh")).read()
    m = re.search(r"constexpr int %s = ([^;]+);" % name, src)
    return m.group(1)


@pytest.mark.parametrize("numel,n,block", _random_plan_configs(200, 2024)[::4] + [([340_000_000], 16, 0),
                                                                                  ([1 << 20, 5, 33], 128, 0)],
                         ids=lambda v: None if not isinstance(v, list) else f"T{len(v)}")
def test_staged_server_copy_windows_stay_in_bounds(numel, n, block):
    """The staged server's bulk copies, recomputed on the host from the plan and the kernel's own
    constants, for every tile of every chunk.  Each worker's sign bytes are copied as a window
    widened to 16-byte boundaries, and each tile's a values as whole 32-element words.  Both must
    stay inside the worker's sign row (stride Wr words) and the padded state, meet the bulk-copy
    rules (16-byte aligned addresses, sizes in multiples of 16), and fit the stage's row slot."""
    kTile = int(_kernel_constant("kTile"))
    expr = _kernel_constant("kRowBytes").replace("kTile", str(kTile))
    assert re.fullmatch(r"[0-9+*/ ()]+", expr), expr
    kRowBytes = int(eval(expr.replace("/", "//"), {"__builtins__": {}}))
    rows = ob.plan_chunks(ob.make_config(numel, n, scale_block=block))
    Dp = sum((L + 31) // 32 * 32 for L in numel)
    Wp = Dp // 32
    Wr = (Wp + 3) // 4 * 4
    for (_, _, _, length, off) in rows:
        for e0 in range(0, length, kTile):
            tlen = min(kTile, length - e0)
            # a: ceil(tlen / 32) words of 32 floats from element off + e0
            a0, abytes = (off + e0) * 4, (tlen + 31) // 32 * 32 * 4
            assert a0 % 16 == 0 and abytes % 16 == 0 and (off + e0) + abytes // 4 <= Dp
            assert abytes <= kTile * 4
            # every worker's sign bytes, widened to a 16-byte window inside its row
            byte0, nb = (off + e0) >> 3, (tlen + 7) // 8
            wlo = byte0 & ~15
            wlen = ((byte0 & 15) + nb + 15) & ~15
            assert wlo % 16 == 0 and wlen % 16 == 0 and (Wr * 4) % 16 == 0
            assert wlo + wlen <= Wr * 4
            assert wlen <= kRowBytes and (byte0 & 15) + nb <= wlen


def test_binding_constants_and_config_layout_match_the_header(tmp_path):
    """The binding restates the header's enums and its config struct for ctypes.  A C program built
    against the header prints the values, the struct's size and every field's offset; they must
    equal the binding's."""
    import shutil
    import subprocess

    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    enums = {
        "ONEBIT_OK": ob.OK, "ONEBIT_ERR_INVALID_ARG": ob.ERR_INVALID_ARG, "ONEBIT_ERR_PHASE": ob.ERR_PHASE,
        "ONEBIT_ERR_CUDA": ob.ERR_CUDA, "ONEBIT_ERR_NOMEM": ob.ERR_NOMEM, "ONEBIT_ERR_WORKSPACE": ob.ERR_WORKSPACE,
        "ONEBIT_ERR_NONFINITE": ob.ERR_NONFINITE, "ONEBIT_ERR_UNSUPPORTED": ob.ERR_UNSUPPORTED,
        "ONEBIT_ERR_BOUNDS": ob.ERR_BOUNDS,
        "ONEBIT_F32": ob.F32, "ONEBIT_F16": ob.F16, "ONEBIT_BF16": ob.BF16,
        "ONEBIT_PHASE_WARMUP": ob.PHASE_WARMUP, "ONEBIT_PHASE_COMPRESS": ob.PHASE_COMPRESS,
        "ONEBIT_STATE_M": ob.STATE_M, "ONEBIT_STATE_V": ob.STATE_V, "ONEBIT_STATE_WORKER_ERROR": ob.STATE_WORKER_ERROR,
        "ONEBIT_STATE_SERVER_ERROR": ob.STATE_SERVER_ERROR, "ONEBIT_STATE_WORKER_BITS": ob.STATE_WORKER_BITS,
        "ONEBIT_STATE_SERVER_BITS": ob.STATE_SERVER_BITS, "ONEBIT_STATE_WORKER_SCALES": ob.STATE_WORKER_SCALES,
        "ONEBIT_STATE_SERVER_SCALES": ob.STATE_SERVER_SCALES,
        "ONEBIT_FAULT_NONE": ob.FAULT_NONE, "ONEBIT_FAULT_STALL_COPIES": ob.FAULT_STALL_COPIES,
        "ONEBIT_FAULT_FAIL_ALLOC": ob.FAULT_FAIL_ALLOC, "ONEBIT_FAULT_TIGHTEN_BOUNDS": ob.FAULT_TIGHTEN_BOUNDS,
        "ONEBIT_NUM_KERNELS": ob.NUM_KERNELS,
    }
    kernels = ["WARMUP", "FREEZE", "WORKER", "WORKER_SCALE", "SERVER", "SERVER_SCALE", "UPDATE", "EXPORT", "EC_UPDATE", "EXCHANGE"]
    for k, name in enumerate(kernels):
        enums[f"ONEBIT_K_{name}"] = ob.KERNEL_NAMES.index(name.lower())
    fields = [f[0] for f in ob.Config._fields_]
    lines = [f'  printf("{e} %d\\n", (int){e});' for e in enums]
    lines.append('  printf("sizeof %zu\\n", sizeof(onebit_adam_config_t));')
    lines += [f'  printf("{f} %zu\\n", offsetof(onebit_adam_config_t, {f}));' for f in fields]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "onebit_adam.h"\nint main(void) {\n'
                   + "\n".join(lines) + "\n  return 0;\n}\n")
    exe = tmp_path / "layout"
    r = subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True).stdout.splitlines())
    for e, v in enums.items():
        assert int(got[e]) == v, e
    assert int(got["sizeof"]) == ctypes.sizeof(ob.Config)
    for f in fields:
        assert int(got[f]) == getattr(ob.Config, f).offset, f
