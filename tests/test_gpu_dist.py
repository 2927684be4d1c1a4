"""The multi-GPU form on the GPU: ranks' handles against one GPU simulating all n workers.

The step is split at the exchange ("1-bit Adam ...", Sec. 6 and Sec. 11 steps 1-3; the AIMech page's
gather-then-broadcast): ``compress_begin`` (this rank's workers), an all-to-all, ``compress_serve``
(this rank's shards), an all-gather, ``compress_end`` (broadcast and update).  Every rank's results
must be bit-identical to the single-GPU handle, which is itself compared with the oracle here
(``parity_util.Pair``) after every step.

Two arrangements, neither of which has kernels waiting on one another across ranks:
  * the ranks' handles in one process on one GPU, the collectives emulated by copying the blocks
    between their buffers (exactly what an all-to-all and an all-gather deliver);
  * two processes sharing the GPU, each one rank, the buffers moved by the package's host-staged
    transport over a gloo process group -- the code path a multi-GPU job runs, with gloo in place of
    NCCL.
"""
import os
import socket

import numpy as np
import pytest
import torch

import communication_compressed_optimizer_compress_gb300 as ob
from communication_compressed_optimizer_compress_gb300 import dist as D
from communication_compressed_optimizer_compress_gb300 import workloads as W
from parity_util import Pair

pytestmark = pytest.mark.gpu

CASES = {
    "ragged_n4_r2_f32": dict(numel=(70_001, 33, 0, 5000, 4099), n=4, R=2, dtype=W.F32, block=0),
    "flat_n16_r16_bf16": dict(numel=(300_007,), n=16, R=16, dtype=W.BF16, block=0),   # one worker per rank
    "flat_n16_r4_f16": dict(numel=(3 * (1 << 20) + 333,), n=16, R=4, dtype=W.F16, block=0),  # staged server
    "blocks_n8_r4_f16": dict(numel=(20_000, 77, 4096), n=8, R=4, dtype=W.F16, block=96),
    "n3_r3_f32": dict(numel=(1000, 31), n=3, R=3, dtype=W.F32, block=0),
    "rank_of_one_n4": dict(numel=(50_000,), n=4, R=1, dtype=W.F32, block=0),
    # 8192-element server chunks (two staged tiles each) in every rank's narrowed chunk table
    "flat_n16_r4_f16_d8M": dict(numel=(8_000_037,), n=16, R=4, dtype=W.F16, block=0),
    # per-block scales at size: the staged server's walk over contiguous runs of a rank's own chunks
    "blocks_n16_r2_bf16_d6M": dict(numel=(6_000_011,), n=16, R=2, dtype=W.BF16, block=65536),
}


def _state(opt, workers):
    out = {"m": opt.export_state(ob.STATE_M), "v": opt.export_state(ob.STATE_V),
           "sb": opt.export_state(ob.STATE_SERVER_BITS), "ws": opt.export_state(ob.STATE_WORKER_SCALES),
           "ss": opt.export_state(ob.STATE_SERVER_SCALES), "se": opt.export_state(ob.STATE_SERVER_ERROR),
           "x": torch.cat([p.detach().reshape(-1) for p in opt.params])}
    for i in workers:
        out[f"d{i}"] = opt.export_state(ob.STATE_WORKER_ERROR, i)
        out[f"b{i}"] = opt.export_state(ob.STATE_WORKER_BITS, i)
    return out


def _own_mask(numel, n, block, R, r):
    """Elements of the shards rank r serves (the per-block segments when block > 0)."""
    import oracle

    segs = oracle.scale_blocks(numel, block)
    nl = n // R
    mask = []
    for L in segs:
        m = np.zeros(L, bool)
        for j in range(r * nl, (r + 1) * nl):
            lo, hi = oracle.shard(L, n, j)
            m[lo:hi] = True
        mask.append(m)
    return torch.from_numpy(np.concatenate(mask) if mask else np.zeros(0, bool)).cuda()


def _same(a, b):
    return torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a,
                       b.view(torch.int32) if b.dtype == torch.float32 else b)


@pytest.mark.parametrize("case", list(CASES))
def test_ranks_in_one_process_match_one_gpu(case):
    c = CASES[case]
    n, R, block = c["n"], c["R"], c["block"]
    nl = n // R
    T = len(c["numel"])
    w = W.WORKLOADS["tiny"].with_(numel=c["numel"], n_workers=n, grad_dtype=c["dtype"], warmup_steps=2,
                                  compress_steps=3, seed=401 + n + R)
    p = Pair(w, scale_block=block)  # the single-GPU handle, compared with the oracle after every step
    x0 = [t.cuda() for t in W.params(w, "cpu")]
    ranks = [D.RankOneBitAdam([t.clone() for t in x0], n, w.warmup_steps, r, R, transport=D.LocalTransport(),
                              beta1=w.beta1, beta2=w.beta2, eps=w.eps, lr=w.lr, grad_dtype=W.TORCH_DTYPE[c["dtype"]],
                              scale_block=block) for r in range(R)]
    masks = [_own_mask(c["numel"], n, block, R, r) for r in range(R)]
    for step in range(2 + 3):
        g = p.grads()
        gd = [t.cuda() for t in g]
        if step < 2:
            p.gpu.warmup_step(gd)
            p.ora.warmup_step([W.to_numpy_grad(t) for t in g])
            p.check_warmup(exact=True)
            for o in ranks:
                ob.OneBitAdam.warmup_step(o, gd)  # every worker's gradient: the warm-up's all-gather done
            continue
        if step == 2:
            p.freeze()
            for o in ranks:
                o.freeze_variance()
        p.gpu.compress_step(gd)
        p.ora.compress_step([W.to_numpy_grad(t) for t in g])
        p.check_compress()
        for r, o in enumerate(ranks):
            o.begin(gd[r * nl * T:(r + 1) * nl * T])
        if R > 1:  # the all-to-all: block q of rank p's send buffer is block p of rank q's receive buffer
            for q, o in enumerate(ranks):
                o.recv.view(R, -1).copy_(torch.stack([ranks[pp].send.view(R, -1)[q] for pp in range(R)]))
        for o in ranks:
            o.serve()
        if R > 1:  # the all-gather
            cat = torch.cat([o.bcast for o in ranks])
            for o in ranks:
                o.gathered.copy_(cat)
        for o in ranks:
            o.end()
        torch.cuda.synchronize()
        want = _state(p.gpu, range(n))
        for r, o in enumerate(ranks):
            assert o.get_status() == ob.OK and o.get_step() == p.gpu.get_step()
            mine = range(r * nl, (r + 1) * nl)
            got = _state(o, mine)
            for k in ("m", "v", "sb", "ws", "ss", "x"):
                assert _same(got[k], want[k]), (case, step, r, k)
            for i in mine:
                assert _same(got[f"d{i}"], want[f"d{i}"]) and _same(got[f"b{i}"], want[f"b{i}"]), (case, step, r, i)
            se = got["se"]  # this rank's shards carry its server error; the rest read 0
            assert _same(se[masks[r]], want["se"][masks[r]]), (case, step, r)
            if R > 1:
                assert bool((se[~masks[r]] == 0).all()), (case, step, r)
    for o in ranks:
        o.free()
    p.close()


def test_split_step_errors():
    """Order and form checks of the split step: on a single-GPU handle the split calls are refused; on
    a rank handle the fused step is refused when world > 1, and the calls must come in order."""
    w = W.WORKLOADS["tiny"].with_(numel=(5000,), n_workers=4, warmup_steps=1, seed=411)
    x0 = [t.cuda() for t in W.params(w, "cpu")]
    g = [t.cuda() for t in W.GradSource(w, "cpu").grads(0)]
    single = ob.OneBitAdam([t.clone() for t in x0], 4, 1)
    single.warmup_step(g)
    single.freeze_variance()
    L = D._lib()
    assert L.onebit_adam_compress_serve(single.h, None, None, None) == ob.ERR_UNSUPPORTED
    o = D.RankOneBitAdam([t.clone() for t in x0], 4, 1, 1, 2, transport=D.LocalTransport())
    ob.OneBitAdam.warmup_step(o, g)  # every worker's gradient (the warm-up's all-gather done)
    with pytest.raises(ob.OneBitError) as e:
        o.begin(g[2:4])  # before the freeze
    assert e.value.status == ob.ERR_PHASE
    o.freeze_variance()
    with pytest.raises(ob.OneBitError) as e:
        o.serve()  # before begin
    assert e.value.status == ob.ERR_PHASE
    with pytest.raises(ob.OneBitError) as e:
        ob.OneBitAdam.compress_step(o, g)  # the fused step needs the exchange
    assert e.value.status == ob.ERR_UNSUPPORTED
    with pytest.raises(ob.OneBitError) as e:
        o.export_state(ob.STATE_WORKER_ERROR, 0)  # worker 0 belongs to rank 0
    assert e.value.status == ob.ERR_INVALID_ARG
    o.begin(g[2:4])
    with pytest.raises(ob.OneBitError) as e:
        o.begin(g[2:4])  # twice
    assert e.value.status == ob.ERR_PHASE
    with pytest.raises(ValueError):
        D.RankOneBitAdam([t.clone() for t in x0], 4, 1, 0, 3)  # 4 workers do not split over 3 ranks
    torch.cuda.synchronize()
    o.free()
    single.free()


# ---------------------------------------------------------------------------------- two processes

def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _proc_main(rank, world, port, numel, n, dtype):
    import torch.distributed as tdist

    tdist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        nl, T = n // world, len(numel)
        w = W.WORKLOADS["tiny"].with_(numel=numel, n_workers=n, grad_dtype=dtype, warmup_steps=2, seed=421)
        src = W.GradSource(w, "cpu")
        x0 = [t.cuda() for t in W.params(w, "cpu")]
        tdt = W.TORCH_DTYPE[dtype]
        ref = ob.OneBitAdam([t.clone() for t in x0], n, 2, grad_dtype=tdt)
        o = D.RankOneBitAdam([t.clone() for t in x0], n, 2, rank, world, transport=D.HostTransport(), grad_dtype=tdt)
        for step in range(5):
            g = [t.cuda() for t in src.grads(step)]
            local = g[rank * nl * T:(rank + 1) * nl * T]
            if step < 2:
                ref.warmup_step(g)
                o.warmup_step(local)  # all-gather of the ranks' gradients over gloo
                continue
            if step == 2:
                ref.freeze_variance()
                o.freeze_variance()
            ref.compress_step(g)
            o.compress_step(local)
            torch.cuda.synchronize()
            a = _state(ref, range(rank * nl, (rank + 1) * nl))
            b = _state(o, range(rank * nl, (rank + 1) * nl))
            for k in ("m", "v", "sb", "ws", "ss", "x"):
                assert _same(a[k], b[k]), (rank, step, k)
            for i in range(rank * nl, (rank + 1) * nl):
                assert _same(a[f"d{i}"], b[f"d{i}"]) and _same(a[f"b{i}"], b[f"b{i}"]), (rank, step, i)
        assert o.get_status() == ob.OK
        o.free()
        ref.free()
    finally:
        tdist.destroy_process_group()


@pytest.mark.parametrize("numel,n,dtype", [((70_001, 33, 5000), 4, W.F16), ((200_003,), 2, W.BF16)],
                         ids=["ragged_n4", "flat_n2"])
def test_two_processes_share_the_gpu(numel, n, dtype):
    import torch.multiprocessing as mp

    mp.spawn(_proc_main, args=(2, _free_port(), numel, n, dtype), nprocs=2, join=True)


def _leave_main(rank, world, port):
    import datetime
    import time

    import torch.distributed as tdist

    tdist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world,
                             timeout=datetime.timedelta(seconds=15))
    torch.cuda.set_device(0)
    n, T = 2, 1
    w = W.WORKLOADS["tiny"].with_(numel=(50_000,), n_workers=n, warmup_steps=2, seed=431)
    src = W.GradSource(w, "cpu")
    o = D.RankOneBitAdam([t.cuda() for t in W.params(w, "cpu")], n, 2, rank, world, transport=D.HostTransport())
    for step in range(4):
        local = [t.cuda() for t in src.grads(step)][rank * T:(rank + 1) * T]
        if step < 2:
            o.warmup_step(local)
            continue
        if step == 2:
            o.freeze_variance()
        o.compress_step(local)
    ckpt = o.state_dict()
    torch.cuda.synchronize()
    tdist.barrier()
    if rank == 1:  # leaves between steps: none of its kernels or collectives in flight
        o.free()
        return
    local = [t.cuda() for t in src.grads(4)][:T]
    t0 = time.time()
    with pytest.raises(D.ExchangeError):
        o.compress_step(local)  # the all-to-all fails: the peer is gone
    assert time.time() - t0 < 90
    assert o.get_step() == (ckpt["t"], ob.PHASE_COMPRESS)  # the step did not count
    o.load_state_dict(ckpt)
    again = o.state_dict()
    torch.cuda.synchronize()
    assert o.get_status() == ob.OK
    for k in ("m", "v", "server_error"):
        assert _same(again[k], ckpt[k]), k
    assert _same(again["worker_error"][0], ckpt["worker_error"][0])
    o.free()
    try:
        tdist.destroy_process_group()
    except Exception:
        pass


def test_a_rank_that_leaves_is_reported_and_the_state_restores():
    """Failure detection of the multi-GPU form without a GPU fault: one rank leaves between steps;
    the other's next step fails in its collective within the process group's timeout, the library
    leaves the split step (ExchangeError), and the rank's checkpoint restores its state bit for bit."""
    import torch.multiprocessing as mp

    mp.spawn(_leave_main, args=(2, _free_port()), nprocs=2, join=True)
