"""The checked build on the GPU: the library compiled with -DONEBIT_CHECKS, whose kernels check each
unit of work (chunk, scale range, exchange range) against their buffers before touching it and
report instead of touching any that would leave them.

* ``test_checked_build_passes_the_parity_cases`` builds the checked library and re-runs a selection
  of the oracle parity cases (tiny to 12e6 elements, chunks up to 40960 elements), the
  grid-independence cases and the multi-GPU form's ranks in a child process that loads it
  (``ONEBIT_LIBRARY=checked``).  Those tests assert ``get_status() == OK``
  after their steps, so every kernel's checks pass on every schedule they run, and their results
  still match the oracle (or, for the ranks, the single handle) bit for bit or within the parity
  protocol.
* ``test_tightened_bounds_are_reported`` (checked library only) narrows the extent the checks allow
  with the ONEBIT_FAULT_TIGHTEN_BOUNDS hook: the units reaching into the withheld end of the rows
  are skipped and reported, the state they cover is left alone, and after the hook is turned off the
  handle steps cleanly again.  The hook only makes the checks stricter, so no access ever leaves
  the buffers.
* ``test_normal_build_has_no_checks``: the same hook is refused by the normal library.
"""
import os
import re
import subprocess
import sys

import pytest
import torch

import communication_compressed_optimizer_compress_gb300 as ob
from communication_compressed_optimizer_compress_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SELECTION = [
    "tests/test_gpu_parity.py::test_tiny_schedule",
    "tests/test_gpu_parity.py::test_odd_sizes",
    "tests/test_gpu_parity.py::test_scale_blocks",
    "tests/test_gpu_parity.py::test_results_do_not_depend_on_the_grid",
    "tests/test_gpu_parity.py::test_ec_adam_baseline_then_compression",
    "tests/test_gpu_parity.py::test_checkpoint_resume",
    "tests/test_gpu_parity.py::test_host_gradient_entry_points",
    "tests/test_gpu_parity.py::test_variance_norm_monitor_matches_oracle",
    "tests/test_gpu_parity.py::test_degenerate_inputs",
    "tests/test_gpu_dist.py::test_ranks_in_one_process_match_one_gpu",
    "tests/test_gpu_parity_large.py::test_large_chunks",
    "tests/test_gpu_checked_build.py::test_tightened_bounds_are_reported",
]


@pytest.mark.skipif(ob.CHECKED, reason="runs the checked library in a child process")
def test_checked_build_passes_the_parity_cases():
    from communication_compressed_optimizer_compress_gb300 import _build

    lib = _build.build(checked=True)
    assert lib.endswith("libonebit_adam_checked.so")
    env = dict(os.environ, ONEBIT_LIBRARY="checked")
    r = subprocess.run([sys.executable, "-m", "pytest", *SELECTION, "-m", "gpu", "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = (r.stdout + r.stderr)[-4000:]
    assert r.returncode == 0, tail
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and int(m.group(1)) >= 86 and "skipped" not in r.stdout, tail  # every selected case ran


def _opt(w):
    params = [p.cuda() for p in W.params(w, "cpu")]
    return ob.OneBitAdam(params, w.n_workers, w.warmup_steps, w.beta1, w.beta2, w.eps, w.lr,
                         grad_dtype=W.TORCH_DTYPE[w.grad_dtype]), params


def _message(opt):
    return ob.lib().onebit_adam_last_error(opt.h).decode()


@pytest.mark.skipif(not ob.CHECKED, reason="needs the checked library (ONEBIT_LIBRARY=checked)")
@pytest.mark.parametrize("numel,n,dtype", [((100_000,), 16, W.F16), ((70_001, 33, 0, 5000), 3, W.F32)],
                         ids=["flat_n16_f16_staged", "ragged_n3_f32_runs"])
def test_tightened_bounds_are_reported(numel, n, dtype):
    w = W.WORKLOADS["tiny"].with_(numel=numel, n_workers=n, grad_dtype=dtype, warmup_steps=2, seed=171)
    src = W.GradSource(w, "cpu")
    g = [[t.cuda() for t in src.grads(s)] for s in range(8)]
    opt, params = _opt(w)

    # warm-up with the last word of the rows withheld: the chunk that reaches it is skipped
    opt.set_fault_injection(ob.FAULT_TIGHTEN_BOUNDS, 32)
    before = torch.cat([p.detach().reshape(-1) for p in params]).clone()
    opt.warmup_step(g[0])
    assert opt.get_status() == ob.ERR_BOUNDS
    assert "warmup" in _message(opt)
    after = torch.cat([p.detach().reshape(-1) for p in params])
    assert torch.equal(after[-1:], before[-1:])    # the skipped chunk's parameters are untouched
    assert not torch.equal(after[:1000], before[:1000])  # the others moved
    opt.set_fault_injection(ob.FAULT_NONE)
    opt.clear_status()
    opt.warmup_step(g[1])
    assert opt.get_status() == ob.OK

    opt.freeze_variance()
    opt.compress_step(g[2])
    opt.compress_step(g[3])
    assert opt.get_status() == ob.OK

    # a compression step: worker, server and update kernels all skip the last chunk
    opt.set_fault_injection(ob.FAULT_TIGHTEN_BOUNDS, 32)
    before = torch.cat([p.detach().reshape(-1) for p in params]).clone()
    opt.compress_step(g[4])
    assert opt.get_status() == ob.ERR_BOUNDS
    msg = _message(opt)
    for k in ("worker", "server", "update"):
        assert k in msg, msg
    after = torch.cat([p.detach().reshape(-1) for p in params])
    assert torch.equal(after[-1:], before[-1:])
    assert not torch.equal(after[:1000], before[:1000])

    # the hook off and the flag cleared, the handle steps cleanly again
    opt.set_fault_injection(ob.FAULT_NONE)
    opt.clear_status()
    opt.compress_step(g[5])
    assert opt.get_status() == ob.OK
    for bad in (0, 31, 33):
        with pytest.raises(ob.OneBitError) as e:
            opt.set_fault_injection(ob.FAULT_TIGHTEN_BOUNDS, bad)
        assert e.value.status == ob.ERR_INVALID_ARG
    opt.free()


@pytest.mark.skipif(ob.CHECKED, reason="the normal library")
def test_normal_build_has_no_checks():
    w = W.WORKLOADS["tiny"].with_(numel=(1000,), n_workers=2, warmup_steps=1)
    opt, _ = _opt(w)
    with pytest.raises(ob.OneBitError) as e:
        opt.set_fault_injection(ob.FAULT_TIGHTEN_BOUNDS, 32)
    assert e.value.status == ob.ERR_UNSUPPORTED
    opt.free()
