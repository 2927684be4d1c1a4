"""CUDA path vs the oracle, element by element, on seeded inputs (free-running; see parity_util)."""
import numpy as np
import pytest
import torch

import communication_compressed_optimizer_compress_gb300 as ob
from communication_compressed_optimizer_compress_gb300 import workloads as W
from parity_util import Pair, _close

pytestmark = pytest.mark.gpu


def _tiny(**kw):
    return W.WORKLOADS["tiny"].with_(**kw)


def test_tiny_schedule():
    """The Tiny workload: 2^20 fp32, n=4, 5 warm-up Adam steps then 5 compression steps, compared
    after every step; the warm-up is bit-exact."""
    p = Pair(_tiny())
    for _ in range(5):
        p.warmup(check=False)
        p.check_warmup(exact=True)
    p.freeze()
    for _ in range(5):
        p.compress()
    st = p.stats
    assert st.excluded_worker <= 1e-6 * st.worker_draws, st
    assert st.scales_exact >= 0.99 * st.scales, st
    p.close()


ODD = [
    ([1], 1), ([31], 2), ([33], 3), ([32 * 4 - 1], 4), ([32 * 4 + 1], 4), ([(1 << 20) + 7], 8),
    ([1, 5, 32, 33], 3), ([5, 0, 33, 200], 4), ([65536 * 2 + 100, 7], 16), ([1000], 16),
    ([5000, 37], 20), ([3000, 2049], 33), ([777, 4100], 32), ([1000, 65], 17), ([300, 1], 256),
    ([5000], 128), ([2000], 200),
]


@pytest.mark.parametrize("numel,n", ODD, ids=[f"{'-'.join(map(str, a))}_n{b}" for a, b in ODD])
@pytest.mark.parametrize("dtype", [W.F32, W.F16, W.BF16], ids=["f32", "f16", "bf16"])
def test_odd_sizes(numel, n, dtype):
    """Ragged tensors, tails that are not a multiple of 8 or 32, empty tensors and shards, several
    chunks per shard, worker counts that are not powers of two, all gradient dtypes.  The worker
    counts cover the server's paths: table only (n <= 12), table + ordered float4 adds (13..16),
    further workers added one by one (17..128, staged kernel, strided or over contiguous runs for
    short-tensor lists), the register kernel (129..256, strided on one flat buffer, contiguous runs on
    short-tensor lists), and the library's maximum n = 256."""
    w = _tiny(numel=tuple(numel), n_workers=n, grad_dtype=dtype, warmup_steps=2, compress_steps=3,
              seed=7 + n + len(numel))
    p = Pair(w)
    st = p.run()
    assert st.scales_exact >= 0.99 * st.scales, st
    p.close()


@pytest.mark.parametrize("dtype", [W.F32, W.F16, W.BF16], ids=["f32", "f16", "bf16"])
def test_misaligned_pointers(dtype):
    """Parameters and gradients that start 4 or 2 bytes into an allocation take the scalar path."""
    w = _tiny(numel=(5000, 77), n_workers=3, grad_dtype=dtype, warmup_steps=2, compress_steps=3, seed=21)
    p = Pair(w, misalign=True)
    p.run()
    p.close()


def test_bias_correction():
    w = _tiny(numel=(4099,), n_workers=2, warmup_steps=4, compress_steps=3, seed=31)
    p = Pair(w, bias_correction=True)
    for _ in range(4):
        p.warmup(check=False)
        p.check_warmup(exact=True)
    p.freeze()
    for _ in range(3):
        p.compress()
    p.close()


def test_heavy_tail_bf16():
    """GPT-2-like gradient law (1% of coordinates x100) in bf16, n=4."""
    w = W.WORKLOADS["gpt2_1p5b"].with_(numel=(300_001,), warmup_steps=3, compress_steps=4)
    p = Pair(w)
    p.run()
    p.close()


def test_block_sigma_f16():
    """BERT-Large-like gradient law (log-uniform per-block sigma) in fp16, n=16, several blocks."""
    w = W.WORKLOADS["bert_large"].with_(numel=(3 * (1 << 20) + 333,), warmup_steps=3, compress_steps=3)
    p = Pair(w)
    p.run()
    p.close()


def _state(opt, n):
    out = {"m": opt.export_state(ob.STATE_M), "v": opt.export_state(ob.STATE_V),
           "eps": opt.export_state(ob.STATE_SERVER_ERROR), "sb": opt.export_state(ob.STATE_SERVER_BITS),
           "ws": opt.export_state(ob.STATE_WORKER_SCALES), "ss": opt.export_state(ob.STATE_SERVER_SCALES)}
    for i in range(n):
        out[f"d{i}"] = opt.export_state(ob.STATE_WORKER_ERROR, i)
        out[f"b{i}"] = opt.export_state(ob.STATE_WORKER_BITS, i)
    return {k: v.cpu().numpy().copy() for k, v in out.items()}


def test_determinism():
    """Two runs on the same inputs give bitwise-identical state (fixed-order reductions)."""
    w = _tiny(numel=(200_003, 4096), n_workers=5, warmup_steps=2, compress_steps=3, seed=41)
    res = []
    for _ in range(2):
        p = Pair(w)
        for _ in range(2):
            p.warmup(check=False)
        p.freeze(check=False)
        for _ in range(3):
            p.compress(check=False)
        torch.cuda.synchronize()
        s = _state(p.gpu, w.n_workers)
        s["x"] = p.x()
        res.append(s)
        p.close()
    for k in res[0]:
        assert np.array_equal(res[0][k].view(np.uint8), res[1][k].view(np.uint8)), k


@pytest.mark.parametrize("block", [0, 96], ids=["per_tensor", "blocks_96"])
def test_checkpoint_resume(block):
    """Export the state after some steps, import it into a fresh handle, continue: the result is
    identical to the uninterrupted run (also with per-block scales, whose exports are per block)."""
    w = _tiny(numel=(70_001, 33), n_workers=3, warmup_steps=2, compress_steps=4, seed=51)
    ref = Pair(w, scale_block=block)
    for _ in range(2):
        ref.warmup(check=False)
    ref.freeze(check=False)
    for _ in range(2):
        ref.compress(check=False)
    torch.cuda.synchronize()
    snap = {k: torch.from_numpy(v).cuda() for k, v in _state(ref.gpu, w.n_workers).items()}
    x_snap = [p.detach().clone() for p in ref.params]
    for _ in range(2):
        ref.compress(check=False)
    torch.cuda.synchronize()
    want = _state(ref.gpu, w.n_workers)
    want_x = ref.x()

    params = [x.clone() for x in x_snap]
    opt = ob.OneBitAdam(params, w.n_workers, w.warmup_steps, w.beta1, w.beta2, w.eps, w.lr, scale_block=block)
    opt.set_step(2 + 2, ob.PHASE_COMPRESS)
    opt.import_state(ob.STATE_V, snap["v"])
    opt.import_state(ob.STATE_M, snap["m"])
    opt.import_state(ob.STATE_SERVER_ERROR, snap["eps"])
    for i in range(w.n_workers):
        opt.import_state(ob.STATE_WORKER_ERROR, snap[f"d{i}"], i)
    src = W.GradSource(w, "cpu")
    for step in (4, 5):
        opt.compress_step([g.cuda() for g in src.grads(step)])
    torch.cuda.synchronize()
    got = _state(opt, w.n_workers)
    got_x = torch.cat([p.cpu() for p in params]).numpy()
    assert np.array_equal(got_x.view(np.uint32), want_x.view(np.uint32))
    for k in want:
        assert np.array_equal(got[k].view(np.uint8), want[k].view(np.uint8)), k
    opt.free()
    ref.close()


@pytest.mark.parametrize("block", [0, 4096], ids=["per_tensor", "blocks_4096"])
def test_host_gradient_entry_points(block):
    """warmup_step_host / compress_step_host (host buffers copied by the library) equal the
    device-pointer entry points, also when the library cuts the tensors into scale blocks after
    staging them."""
    w = _tiny(numel=(10_007, 64), n_workers=2, grad_dtype=W.F16, warmup_steps=2, compress_steps=2, seed=61)
    a, b = Pair(w, scale_block=block), Pair(w, scale_block=block)
    for step in range(4):
        g = a.grads()
        b.grads()
        host = [t.pin_memory() for t in g]
        dev = [t.cuda() for t in g]
        if step < 2:
            a.gpu.warmup_step(dev)
            b.gpu.warmup_step_host(host)
        else:
            if step == 2:
                a.gpu.freeze_variance()
                b.gpu.freeze_variance()
            a.gpu.compress_step(dev)
            b.gpu.compress_step_host(host)
    torch.cuda.synchronize()
    assert np.array_equal(a.x().view(np.uint32), b.x().view(np.uint32))
    sa, sb = _state(a.gpu, 2), _state(b.gpu, 2)
    for k in sa:
        assert np.array_equal(sa[k].view(np.uint8), sb[k].view(np.uint8)), k
    a.close()
    b.close()


def test_phase_errors_and_status():
    w = _tiny(numel=(1000,), n_workers=2, warmup_steps=2)
    p = Pair(w)
    g = [t.cuda() for t in p.src.grads(0)]
    with pytest.raises(ob.OneBitError) as e:
        p.gpu.compress_step(g)
    assert e.value.status == ob.ERR_PHASE
    with pytest.raises(ob.OneBitError) as e:
        p.gpu.freeze_variance()  # before any warm-up step
    assert e.value.status == ob.ERR_PHASE
    p.gpu.warmup_step(g)
    p.gpu.warmup_step(g)
    with pytest.raises(ob.OneBitError) as e:
        p.gpu.warmup_step(g)  # T_w reached
    assert e.value.status == ob.ERR_PHASE
    p.gpu.freeze_variance()
    with pytest.raises(ob.OneBitError) as e:
        p.gpu.warmup_step(g)
    assert e.value.status == ob.ERR_PHASE
    p.gpu.compress_step(g)
    assert p.gpu.get_status() == ob.OK
    assert p.gpu.get_step() == (3, ob.PHASE_COMPRESS)
    # a NaN gradient makes that worker's scale non-finite: the sticky flag reports it
    bad = [t.clone() for t in g]
    bad[1][17] = float("nan")
    p.gpu.compress_step(bad)
    assert p.gpu.get_status() == ob.ERR_NONFINITE
    p.gpu.clear_status()
    assert p.gpu.get_status() == ob.OK
    p.close()


def test_stalled_copies_are_reported_not_hung():
    """Failure detection without a GPU fault: the staged server kernel is made to wait for bytes
    that never arrive; its bounded wait runs out, the status reports it, and the context still
    works (a later step on a fresh handle is correct)."""
    w = _tiny(numel=(20_000,), n_workers=4, warmup_steps=1, compress_steps=2, seed=81)
    p = Pair(w)
    p.warmup(check=False)
    p.freeze(check=False)
    p.gpu.set_fault_injection(ob.FAULT_STALL_COPIES, 64)
    p.gpu.compress_step([t.cuda() for t in p.src.grads(5)])
    assert p.gpu.get_status() == ob.ERR_CUDA
    assert "timed out" in ob.lib().onebit_adam_last_error(p.gpu.h).decode()
    p.gpu.set_fault_injection(ob.FAULT_NONE)
    p.close()
    q = Pair(w)  # the CUDA context is still usable: a full schedule matches the oracle
    q.run()
    q.close()


def test_allocation_failure_is_reported_and_changes_nothing():
    """Failure detection on the host: refused allocations (the host-gradient staging buffers, the
    variance monitor's pinned slot) come back as ONEBIT_ERR_NOMEM with the step count, phase and
    state untouched; once the hook is cleared the same calls succeed and the run matches the oracle
    bit for bit."""
    w = _tiny(numel=(20_000, 77), n_workers=4, grad_dtype=W.F16, warmup_steps=3, seed=87)
    p = Pair(w)
    p.warmup()  # one device-pointer step first, so that there is state to protect
    before = (p.x().copy(), p.gpu.export_state(ob.STATE_M).cpu().numpy().copy())
    g = p.grads()
    host = [t.contiguous().pin_memory() for t in g]
    p.gpu.set_fault_injection(ob.FAULT_FAIL_ALLOC, 1)
    with pytest.raises(ob.OneBitError) as e:
        p.gpu.warmup_step_host(host)
    assert e.value.status == ob.ERR_NOMEM
    torch.cuda.synchronize()
    assert p.gpu.get_step() == (1, ob.PHASE_WARMUP)
    assert np.array_equal(p.x().view(np.uint32), before[0].view(np.uint32))
    assert np.array_equal(p.gpu.export_state(ob.STATE_M).cpu().numpy().view(np.uint32), before[1].view(np.uint32))
    p.gpu.set_fault_injection(ob.FAULT_FAIL_ALLOC, 1)  # the one refusal above is used up
    with pytest.raises(ob.OneBitError) as e:
        p.gpu.set_variance_monitor(True)
    assert e.value.status == ob.ERR_NOMEM
    p.gpu.set_fault_injection(ob.FAULT_NONE)
    p.gpu.set_variance_monitor(True)
    p.gpu.warmup_step_host(host)
    p.ora.warmup_step([W.to_numpy_grad(t) for t in g])
    p.check_warmup(exact=True)
    p.close()


@pytest.mark.parametrize("numel,n,dtype", [((300_000,), 16, W.F16), ((70_001, 33, 0, 5, 4096), 16, W.F16),
                                           ((50_000, 7), 33, W.BF16), ((60_000,), 129, W.F16)],
                         ids=["flat_n16_staged", "ragged_n16_runs", "n33_runs", "n129_register"])
def test_results_do_not_depend_on_the_grid(numel, n, dtype):
    """The same schedule with every streaming launch capped at 1, 7 or 152 CTAs, or uncapped, leaves
    bit-identical state: partial sums are per chunk and reduced in a fixed order, whatever the grid.
    The cases reach the staged server's strided walk, its walk over contiguous runs (whose split
    depends on the grid), and the register server (n > 128)."""
    w = _tiny(numel=numel, n_workers=n, grad_dtype=dtype, warmup_steps=2, seed=151)
    src = W.GradSource(w, "cpu")
    g = [[t.cuda() for t in src.grads(s)] for s in range(5)]
    results = []
    for cap in (0, 1, 7, 152):
        params = [p.cuda() for p in W.params(w, "cpu")]
        opt = ob.OneBitAdam(params, n, w.warmup_steps, w.beta1, w.beta2, w.eps, w.lr, grad_dtype=W.TORCH_DTYPE[dtype])
        opt.set_max_ctas(cap)
        opt.set_variance_monitor(True)
        opt.warmup_step(g[0])
        opt.warmup_step(g[1])
        vnorm = opt.variance_norm()
        opt.freeze_variance()
        for s in range(2, 5):
            opt.compress_step(g[s])
        torch.cuda.synchronize()
        assert opt.get_status() == ob.OK
        st = _state(opt, n)
        st["x"] = torch.cat(params).cpu().numpy()
        results.append((st, vnorm))
        opt.free()
    ref, ref_norm = results[0]
    for st, vnorm in results[1:]:
        assert vnorm == ref_norm
        for k in ref:
            assert np.array_equal(st[k].view(np.uint8), ref[k].view(np.uint8)), k


def test_guard_bands_untouched():
    """Bounds: parameters, gradients and a caller-owned workspace sit between canary bands; a full
    schedule (warm-up, freeze, compression, host-buffer steps, export) writes none of the bands and
    never writes the gradients."""
    w = _tiny(numel=(70_001, 33, 5, 4096), n_workers=16, grad_dtype=W.F16, warmup_steps=2, seed=161)
    n, T = w.n_workers, w.n_tensors
    G = 4096  # guard elements on each side (keeps 256-byte alignment)
    dev = torch.device("cuda")

    def guarded(values, fill):
        buf = torch.full((values.numel() + 2 * G,), fill, dtype=values.dtype, device=dev)
        buf[G:G + values.numel()].copy_(values.reshape(-1))
        return buf, buf[G:G + values.numel()]

    pbufs, params = zip(*[guarded(p.cuda(), float("nan")) for p in W.params(w, "cpu")])
    ws_bytes = ob.workspace_size(ob.make_config(list(w.numel), n, w.warmup_steps, grad_dtype=ob.F16))
    wsbuf = torch.full((ws_bytes + 2 * G,), 0xA5, dtype=torch.uint8, device=dev)
    opt = ob.OneBitAdam(list(params), n, w.warmup_steps, w.beta1, w.beta2, w.eps, w.lr,
                        grad_dtype=torch.float16, workspace=wsbuf[G:G + ws_bytes])
    src = W.GradSource(w, "cpu")
    gbufs_all = []
    for step in range(6):
        pairs = [guarded(t.cuda(), float("inf")) for t in src.grads(step)]
        gbufs, grads = zip(*pairs)
        before = [b.clone() for b in gbufs]
        if step < 2:
            opt.warmup_step(list(grads))
        elif step < 4:
            if step == 2:
                opt.freeze_variance()
            opt.compress_step(list(grads))
        else:
            opt.compress_step_host([t.cpu().pin_memory() for t in grads])
        torch.cuda.synchronize()
        for b, b0 in zip(gbufs, before):
            assert torch.equal(b.view(torch.int16), b0.view(torch.int16)), "a gradient was written"
        gbufs_all.append(gbufs)
    for what in (ob.STATE_M, ob.STATE_V, ob.STATE_SERVER_ERROR, ob.STATE_SERVER_BITS, ob.STATE_WORKER_SCALES):
        opt.export_state(what)
    torch.cuda.synchronize()
    assert opt.get_status() == ob.OK
    for b in pbufs:
        assert torch.isnan(b[:G]).all() and torch.isnan(b[-G:]).all(), "a parameter guard band was written"
    assert bool((wsbuf[:G] == 0xA5).all()) and bool((wsbuf[-G:] == 0xA5).all()), "a workspace guard band was written"
    opt.free()


@pytest.mark.parametrize("dtype", [W.F32, W.F16], ids=["f32", "f16"])
def test_degenerate_inputs(dtype):
    """Degenerate inputs, compared with the oracle bit for bit: all-zero and all-negative-zero
    gradients (every c and a is a signed zero, every sign bit +1 by the sign(0) = +1 convention, all
    scales 0, x unchanged), then gradients of one magnitude with a fixed sign pattern (compression
    lossless, errors exactly 0)."""
    w = _tiny(numel=(4096 + 13, 77), n_workers=4, grad_dtype=dtype, warmup_steps=2, seed=171)
    p = Pair(w)
    tdt = W.TORCH_DTYPE[dtype]
    rng = np.random.default_rng(7)
    signs = [np.where(rng.random(L) < 0.5, -1.0, 1.0) for L in w.numel]

    def step(grads_np, kind):
        dev = [torch.from_numpy(g).to(tdt).cuda() for g in grads_np]
        host = [W.to_numpy_grad(torch.from_numpy(g).to(tdt)) for g in grads_np]
        if kind == "warmup":
            p.gpu.warmup_step(dev)
            p.ora.warmup_step(host)
        else:
            p.gpu.compress_step(dev)
            p.ora.compress_step(host)

    zeros = [np.zeros(L, np.float32) for L in w.numel] * w.n_workers
    negz = [np.full(L, -0.0, np.float32) for L in w.numel] * w.n_workers
    const = [(s * 2.0 ** -7).astype(np.float32) for s in signs] * w.n_workers
    step(zeros, "warmup")
    step(negz, "warmup")
    p.check_warmup(exact=True)
    p.freeze()
    for g in (zeros, negz, const, const, zeros):
        step(g, "compress")
        p.check_compress()
    assert p.stats.excluded_worker == 0 and p.stats.excluded_server == 0
    # after the zero steps every broadcast bit is +1; the constant steps compress losslessly
    assert np.all(p.gpu.export_state(ob.STATE_WORKER_ERROR, 0).cpu().numpy() == p.ora.view("delta")[0])
    p.close()


@pytest.mark.parametrize("dtype", [W.F32, W.BF16], ids=["f32", "bf16"])
def test_norms_at_extreme_magnitudes(dtype):
    """The scales preserve the magnitude of the compressed vector ("1-bit Adam ...", Sec. 4.3; the
    codewithpapers "1-bit Adam" scale definition) at any magnitude: whole tensors whose gradients,
    and hence c and a, sit near 2^-51, at 1e-20 and 1e-30 (squares far below fp32's subnormal range)
    and at 1e25 (squares beyond fp32's range; v overflows to infinity there, on both sides), beside
    two ordinary tensors.  Every scale must match the oracle's exact double-precision norm within one ulp
    (almost all exactly) and every state element within the parity tolerance."""
    numel = (5000, 4099, 3001, 6000, 2003, 4096 + 7)
    w = _tiny(numel=numel, n_workers=4, grad_dtype=dtype, law="tensor_std",
              tensor_std=(1e-3, 2.0 ** -51, 1e-20, 1e-30, 1e25, 1e-3), warmup_steps=2, compress_steps=3, seed=191)
    p = Pair(w)
    for _ in range(2):
        p.warmup()
    p.freeze()
    for _ in range(3):
        p.compress()
    st = p.stats
    assert st.scales_exact >= 0.95 * st.scales, st
    p.close()


def test_two_handles_on_two_streams():
    """Two optimizers stepped in interleaved order on two non-default CUDA streams (their kernels
    free to overlap) end bit-identical to the same schedules run alone on the default stream: a
    handle owns all its state, and every call runs on the stream it is given."""
    ws = [_tiny(numel=(70_001, 33), n_workers=4, grad_dtype=W.F16, warmup_steps=2, seed=181),
          _tiny(numel=(50_000,), n_workers=16, grad_dtype=W.BF16, warmup_steps=2, seed=182)]
    grads = [[[t.cuda() for t in W.GradSource(w, "cpu").grads(s)] for s in range(5)] for w in ws]

    def make(w):
        params = [p.cuda() for p in W.params(w, "cpu")]
        return params, ob.OneBitAdam(params, w.n_workers, w.warmup_steps, w.beta1, w.beta2, w.eps, w.lr,
                                     grad_dtype=W.TORCH_DTYPE[w.grad_dtype])

    def schedule(opt, g, s, stream):
        if s < 2:
            opt.warmup_step(g[s], stream=stream)
        else:
            if s == 2:
                opt.freeze_variance(stream=stream)
            opt.compress_step(g[s], stream=stream)

    alone = []
    for w, g in zip(ws, grads):
        params, opt = make(w)
        for s in range(5):
            schedule(opt, g, s, None)
        torch.cuda.synchronize()
        alone.append((torch.cat([p.cpu() for p in params]).numpy(), _state(opt, w.n_workers)))
        opt.free()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    made = [make(w) for w in ws]
    for s in range(5):
        for k in (0, 1):
            schedule(made[k][1], grads[k], s, streams[k])
    torch.cuda.synchronize()
    for k, w in enumerate(ws):
        params, opt = made[k]
        x = torch.cat([p.cpu() for p in params]).numpy()
        assert np.array_equal(x.view(np.uint32), alone[k][0].view(np.uint32)), k
        st = _state(opt, w.n_workers)
        for key in st:
            assert np.array_equal(st[key].view(np.uint8), alone[k][1][key].view(np.uint8)), (k, key)
        opt.free()


def test_learning_rate_schedule():
    """gamma changed before every step (a warm-up ramp, then decay) on both sides: parity holds
    step by step, and the warm-up stays bit-exact."""
    w = _tiny(numel=(70_001, 33), n_workers=4, grad_dtype=W.F16, warmup_steps=3, seed=191)
    p = Pair(w)
    lrs = [np.float32(v) for v in (1e-4, 5e-4, 1e-3, 8e-4, 4e-4, 2e-4, 1e-4)]
    for s in range(3):
        p.gpu.set_lr(lrs[s])
        p.ora.set_lr(lrs[s])
        p.warmup(check=False)
        p.check_warmup(exact=True)
    p.freeze()
    for s in range(3, 7):
        p.gpu.set_lr(lrs[s])
        p.ora.set_lr(lrs[s])
        p.compress()
    with pytest.raises(ob.OneBitError):
        p.gpu.set_lr(float("nan"))
    p.close()


@pytest.mark.parametrize("phase", ["compress", "ec_adam"])
def test_state_dict_round_trip(phase):
    """state_dict() taken mid-run and loaded into a fresh handle resumes bit-identically: in the
    compression stage, and in the warm-up phase between gradient-compression baseline steps, whose
    error memories are part of the state."""
    w = _tiny(numel=(70_001, 33), n_workers=3, grad_dtype=W.BF16, warmup_steps=10, seed=201)
    src = W.GradSource(w, "cpu")
    g = [[t.cuda() for t in src.grads(s)] for s in range(8)]

    def step(opt, s):
        if phase == "ec_adam":
            opt.ec_adam_step(g[s])
        elif s < 2:
            opt.warmup_step(g[s])
        else:
            if s == 2:
                opt.freeze_variance()
            opt.compress_step(g[s])

    def make(params):
        return ob.OneBitAdam(params, w.n_workers, w.warmup_steps, w.beta1, w.beta2, w.eps, w.lr,
                             grad_dtype=W.TORCH_DTYPE[w.grad_dtype])

    params = [p.cuda() for p in W.params(w, "cpu")]
    ref = make(params)
    for s in range(4):
        step(ref, s)
    ckpt = ref.state_dict()
    ckpt_x = [p.clone() for p in params]
    for s in range(4, 8):
        step(ref, s)
    torch.cuda.synchronize()
    want = _state(ref, w.n_workers)
    want_x = torch.cat([p.cpu() for p in params]).numpy()

    params2 = [x.clone() for x in ckpt_x]
    opt = make(params2)
    # the import copies asynchronously, so tensors it would have to copy first are refused
    strided = torch.zeros(2 * ckpt["m"].numel(), device="cuda")[::2]
    for bad in (strided, ckpt["m"].cpu()):
        with pytest.raises(ValueError):
            opt.import_state(ob.STATE_M, bad)
    opt.load_state_dict(ckpt)
    for s in range(4, 8):
        step(opt, s)
    torch.cuda.synchronize()
    got = _state(opt, w.n_workers)
    got_x = torch.cat([p.cpu() for p in params2]).numpy()
    assert np.array_equal(got_x.view(np.uint32), want_x.view(np.uint32))
    for k in want:
        assert np.array_equal(got[k].view(np.uint8), want[k].view(np.uint8)), k
    opt.free()
    ref.free()


def test_timing_and_launch_counts():
    w = _tiny(numel=(50_000,), n_workers=4, warmup_steps=1)
    p = Pair(w)
    p.gpu.set_timing(True)
    p.warmup(check=False)
    p.freeze(check=False)
    p.compress(check=False)
    t = p.gpu.kernel_times()
    assert t["warmup"][1] == 1 and t["freeze"][1] == 1
    for k in ("worker", "server", "server_scale", "update"):
        assert t[k][1] == 1 and t[k][0] > 0.0, (k, t[k])
    assert t["worker_scale"][1] == 2 and t["worker_scale"][0] > 0.0  # the partials' range repair, the scales
    n0 = p.gpu.launch_count()
    p.compress(check=False)
    assert p.gpu.launch_count() - n0 == 6
    p.close()


def test_workspace_caller_owned():
    """A caller-provided workspace (torch uint8 tensor) gives the same results as a library one."""
    w = _tiny(numel=(12_345,), n_workers=3, warmup_steps=2, compress_steps=2, seed=71)
    ws_bytes = ob.workspace_size(ob.make_config(list(w.numel), w.n_workers, w.warmup_steps))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    a = Pair(w)
    params = [torch.cat([x.clone() for x in W.params(w, "cpu")]).cuda()]
    opt = ob.OneBitAdam(params, w.n_workers, w.warmup_steps, w.beta1, w.beta2, w.eps, w.lr, workspace=ws)
    src = W.GradSource(w, "cpu")
    for step in range(4):
        g = [t.cuda() for t in src.grads(step)]
        if step < 2:
            opt.warmup_step(g)
            a.warmup(check=False)
        else:
            if step == 2:
                opt.freeze_variance()
                a.freeze(check=False)
            opt.compress_step(g)
            a.compress(check=False)
    torch.cuda.synchronize()
    assert np.array_equal(params[0].cpu().numpy().view(np.uint32), a.x().view(np.uint32))
    with pytest.raises(ob.OneBitError) as e:
        ob.OneBitAdam(params, w.n_workers, w.warmup_steps, workspace=ws[: ws_bytes // 2])
    assert e.value.status == ob.ERR_WORKSPACE
    opt.free()
    a.close()


@pytest.mark.parametrize("n,dtype", [(3, W.F16), (16, W.BF16), (8, W.F32)], ids=["small_batch", "staged", "batched"])
def test_variance_norm_monitor_matches_oracle(n, dtype):
    """||v_t||_2 reported during warm-up equals the oracle's norm of its own v after every step, for
    each form of the warm-up kernel (small register batch, shared-memory staged, register batch)."""
    import oracle

    w = _tiny(numel=(70_001, 333, 5), n_workers=n, grad_dtype=dtype, warmup_steps=4, seed=101 + n)
    p = Pair(w)
    p.gpu.set_variance_monitor(True)
    for t in range(1, 5):
        p.warmup()
        got, step = p.gpu.variance_norm()
        want = oracle.norm2(p.ora.view("v"))
        assert step == t
        assert abs(got - want) <= 1e-12 * want, (t, got, want)
    p.close()


def test_warmup_until_stable_stops_where_the_closed_form_says():
    """Constant gradient: ||v_t|| = (1 - b2^t) ||g^2||, so the relative change per step is
    b2^(t-1) (1 - b2) / (1 - b2^(t-1)); the helper must freeze at the first step where it drops to
    the tolerance."""
    import math

    w = _tiny(numel=(50_000,), n_workers=2, warmup_steps=100, seed=111)
    p = Pair(w)
    g = [t.cuda() for t in p.src.grads(0)]
    b2 = float(np.float32(w.beta2))
    r = {t: b2 ** (t - 1) * (1 - b2) / (1 - b2 ** (t - 1)) for t in range(2, 101)}
    t_star = 21
    tol = math.sqrt(r[t_star] * r[t_star - 1])  # between two consecutive steps' changes
    steps = p.gpu.warmup_until_stable(lambda t: g, tol)
    assert steps == t_star, (steps, t_star)
    assert p.gpu.get_step() == (t_star, ob.PHASE_COMPRESS)
    p.close()


def test_auto_freeze_through_the_c_abi():
    """onebit_adam_set_auto_freeze: the library itself freezes at the first warm-up step whose
    variance-norm change drops to the tolerance (the constant-gradient closed form above), leaving
    den, x and m bit-identical to the oracle's warm-up and freeze; with a tolerance never met it
    freezes at T_w; bad tolerances are refused."""
    import math

    w = _tiny(numel=(50_000,), n_workers=2, warmup_steps=100, seed=111)
    p = Pair(w)
    g_host = p.src.grads(0)
    g = [t.cuda() for t in g_host]
    b2 = float(np.float32(w.beta2))
    r = {t: b2 ** (t - 1) * (1 - b2) / (1 - b2 ** (t - 1)) for t in range(2, 101)}
    t_star = 21
    for bad in (-1.0, float("nan"), float("inf")):
        with pytest.raises(ob.OneBitError) as e:
            p.gpu.set_auto_freeze(bad)
        assert e.value.status == ob.ERR_INVALID_ARG
    p.gpu.set_auto_freeze(math.sqrt(r[t_star] * r[t_star - 1]))
    t = 0
    while p.gpu.get_step()[1] == ob.PHASE_WARMUP:
        p.gpu.warmup_step(g)
        p.ora.warmup_step([W.to_numpy_grad(x) for x in g_host])
        t += 1
    assert t == t_star and p.gpu.get_step() == (t_star, ob.PHASE_COMPRESS)
    p.ora.freeze()
    torch.cuda.synchronize()
    assert np.array_equal(p.gpu.export_state(ob.STATE_V).cpu().numpy().view(np.uint32), p.ora.view("den").view(np.uint32))
    assert np.array_equal(p.x().view(np.uint32), p.ora.view("x").view(np.uint32))
    p.close()

    w2 = _tiny(numel=(5000,), n_workers=2, warmup_steps=3, seed=112)
    q = Pair(w2)
    q.gpu.set_auto_freeze(1e-30)  # never met: the freeze comes at T_w
    for step in range(3):
        assert q.gpu.get_step() == (step, ob.PHASE_WARMUP)
        q.warmup(check=False)
    assert q.gpu.get_step() == (3, ob.PHASE_COMPRESS)
    q.ora.freeze()
    q.gpu.set_auto_freeze(0.0)
    q.compress()  # the compression stage continues from the library's own freeze
    q.close()


@pytest.mark.parametrize("numel,n,dtype,bc", [
    ((1 << 20,), 4, W.F16, True), ((70_001, 33, 0, 5), 3, W.F32, False), ((200_000,), 16, W.BF16, False),
], ids=["flat_f16_bc", "ragged_f32", "n16_bf16"])
def test_ec_adam_baseline_then_compression(numel, n, dtype, bc):
    """The gradient-compression baseline (1-bit EC compression of the gradients, then Adam) against
    the oracle for several steps, then the variance freeze and compression-stage steps: every phase
    transition (errors reset at the freeze, Adam's fp32 momentum feeding the first compression step)
    is compared too."""
    w = _tiny(numel=numel, n_workers=n, grad_dtype=dtype, warmup_steps=10, seed=121 + n)
    p = Pair(w, bias_correction=bc)
    for _ in range(4):
        p.ec_adam()
    p.warmup()
    p.ec_adam()
    p.freeze()
    for _ in range(3):
        p.compress()
    assert p.stats.scales_exact >= 0.99 * p.stats.scales, p.stats
    p.close()


@pytest.mark.parametrize("numel,n,dtype,block", [
    ((1 << 20,), 4, W.F32, 4096), ((70_001, 33, 0, 5), 3, W.F16, 96), ((200_000, 1000), 16, W.BF16, 65536),
    ((5000,), 20, W.F32, 32),
], ids=["flat_f32_b4096", "ragged_f16_b96", "n16_bf16_b65536", "n20_b32"])
def test_scale_blocks(numel, n, dtype, block):
    """Per-chunk scale granularity: every block of `block` elements has its own worker scales and
    server shards.  Blocks shorter than n*32 leave empty shards (block 96 with n = 3 is three shards
    of 32; block 32 with n = 20 is one non-empty shard and 19 empty ones), and the last block of a
    tensor is ragged."""
    w = _tiny(numel=numel, n_workers=n, grad_dtype=dtype, warmup_steps=2, compress_steps=4, seed=141 + n)
    p = Pair(w, scale_block=block)
    T_blocks = len(p.numel)
    st = p.run()
    assert p.gpu.export_state(ob.STATE_WORKER_SCALES).numel() == n * T_blocks
    assert st.scales_exact >= 0.99 * st.scales, st
    ws = p.gpu.export_state(ob.STATE_WORKER_SCALES).cpu().numpy().reshape(n, T_blocks)
    if T_blocks > len(numel):  # the scales really are per block
        assert len(np.unique(ws[0])) > 1
    p.close()


def _random_parity_configs(count, seed):
    """Seeded random lists for the parity sweep: empty, tiny, ragged and multi-chunk tensors, worker
    counts across every server path, all gradient dtypes, per-tensor or per-block scales; a few
    hundred thousand elements at most, so that the oracle keeps up."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        T = int(rng.integers(1, 13))
        kind = rng.choice(4, size=T, p=[0.1, 0.3, 0.35, 0.25])
        lo = np.array([0, 1, 65, 5000])[kind]
        hi = np.array([1, 65, 5000, 60_000])[kind]
        numel = [int(rng.integers(a, b)) for a, b in zip(lo, hi)]
        if not sum(numel):
            numel[-1] = 1
        n = int(rng.choice([1, 2, 3, 5, 8, 13, 16, 17, 20, 33, 64, 129]))
        dtype = int(rng.choice([W.F32, W.F16, W.BF16]))
        block = 0 if rng.random() < 0.6 else 32 * int(rng.integers(1, 513))
        out.append((tuple(numel), n, dtype, block, int(rng.integers(1 << 30))))
    return out


@pytest.mark.parametrize("numel,n,dtype,block,seed", _random_parity_configs(12, 7),
                         ids=[f"r{i}" for i in range(12)])
def test_random_configs(numel, n, dtype, block, seed):
    """The CUDA path against the oracle on seeded random parameter lists: warm-up, freeze and
    compression steps compared after every step, as in the fixed cases."""
    w = _tiny(numel=numel, n_workers=n, grad_dtype=dtype, warmup_steps=2, compress_steps=3, seed=seed)
    p = Pair(w, scale_block=block)
    st = p.run()
    assert st.scales_exact >= 0.99 * st.scales, st
    p.close()


def test_cuda_graph_replay_equals_eager():
    """A compression step enqueues kernels only (no host synchronisation or allocation), so a pair
    of steady-state steps (one full cycle of the double-buffered scales) can be captured in a CUDA
    graph and replayed; every replay equals two eager steps bit for bit.  The gradient-pointer
    tables are cached by the eager steps before the capture."""
    w = _tiny(numel=(100_003, 77), n_workers=4, grad_dtype=W.F16, warmup_steps=2, seed=131)
    a, b = Pair(w), Pair(w)
    g = [[t.cuda() for t in a.src.grads(s)] for s in range(2)]
    for p in (a, b):
        for s in range(2):
            p.gpu.warmup_step(g[s])
        p.gpu.freeze_variance()
        for s in range(4):
            p.gpu.compress_step(g[s % 2])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            a.gpu.compress_step(g[0])
            a.gpu.compress_step(g[1])
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        graph.replay()
        b.gpu.compress_step(g[0])
        b.gpu.compress_step(g[1])
    torch.cuda.synchronize()
    assert np.array_equal(a.x().view(np.uint32), b.x().view(np.uint32))
    sa, sb = _state(a.gpu, w.n_workers), _state(b.gpu, w.n_workers)
    for k in sa:
        assert np.array_equal(sa[k].view(np.uint8), sb[k].view(np.uint8)), k
    a.close()
    b.close()
