"""The multi-GPU form's partition and exchange, on CPU ranks (gloo, world size 2; no GPU).

Each rank plays its part of the step the way the library splits it -- its own workers' compression,
the all-to-all of the packed messages, its own shards' server step, the all-gather of the server
results, the update -- with the oracle's compressor doing the arithmetic ("1-bit Adam ...", Sec. 11
steps 1-3: worker error-compensated compression, server average and recompression, broadcast and
update).  What is under test is the host side of the product: the library's exchange plan
(``onebit_adam_plan_exchange``: which words and scales go into which block, and where they land) and
the Python transport that moves the blocks between ranks (``dist.HostTransport`` over gloo).  After
every step each rank's broadcast, parameters and momentum, its workers' messages and errors, and its
shards' server state must equal the single-process oracle's bit for bit.
"""
import os
import socket

import numpy as np
import pytest
import torch

import oracle
from communication_compressed_optimizer_compress_gb300 import workloads as W

CASES = {
    # ragged tensors with short, empty and multi-word shards; two workers per rank
    "ragged_n4_w2": dict(numel=(100, 33, 0, 700, 4099), n=4, world=2, block=0, dtype=W.F32),
    # one worker per rank (the pages' setup: every GPU is one worker and one server)
    "flat_n2_w2": dict(numel=(5000,), n=2, world=2, block=0, dtype=W.F16),
    # per-block scales: every block is a segment of its own with its own shards
    "blocks_n4_w2": dict(numel=(1000, 77), n=4, world=2, block=96, dtype=W.BF16),
}


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bits(words, L):
    w = np.asarray(words, np.uint32)
    return ((w[:, None] >> np.arange(32, dtype=np.uint32)[None, :]) & 1).astype(bool).reshape(-1)[:L]


def _decode(g):
    h = W.to_numpy_grad(g)
    if h.dtype == np.uint16:
        return (h.astype(np.uint32) << 16).view(np.float32)
    return h.astype(np.float32)


def _apply(rows, stage, regions, buf):
    """Carry out one stage of the plan's copies on host arrays (regions 0-3, buffer = region 4 as a
    [blocks, words] array); scales travel as their bit patterns."""
    for st, sreg, srow, soff, dreg, drow, doff, n in rows:
        if st != stage:
            continue
        src = buf[srow] if sreg == 4 else regions[sreg][srow]
        dst = buf[drow] if dreg == 4 else regions[dreg][drow]
        dst[doff: doff + n] = src[soff: soff + n]


def _rank_main(rank, world, port, case):
    import torch.distributed as tdist

    import communication_compressed_optimizer_compress_gb300 as ob
    from communication_compressed_optimizer_compress_gb300 import dist as D

    tdist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        c = CASES[case]
        n, numel, block, dtype = c["n"], c["numel"], c["block"], c["dtype"]
        nl, w0 = n // world, rank * (n // world)
        w = W.WORKLOADS["tiny"].with_(numel=numel, n_workers=n, grad_dtype=dtype, warmup_steps=2, seed=301)
        segs = oracle.scale_blocks(numel, block)
        T, D_ = len(segs), sum(segs)
        soff = np.concatenate([[0], np.cumsum(segs)]).astype(np.int64)
        woff = np.concatenate([[0], np.cumsum([(L + 31) // 32 for L in segs])]).astype(np.int64)
        Wd = int(woff[-1])
        cfg = ob.make_config(list(numel), n, 2, grad_dtype=dtype, scale_block=block)
        rows, send_block, bcast_block = D.plan_exchange(cfg, rank, world)
        transport = D.HostTransport()

        src = W.GradSource(w, "cpu")
        x0 = torch.cat(W.params(w, "cpu")).numpy()
        ref = oracle.OneBitAdamOracle(list(numel), n, x0, w.beta1, w.beta2, w.eps, w.lr, grad_dtype=dtype,
                                      scale_block=block)
        mine = oracle.OneBitAdamOracle(list(numel), n, x0, w.beta1, w.beta2, w.eps, w.lr, grad_dtype=dtype,
                                       scale_block=block)
        Tu = len(numel)
        # warm-up: the uncompressed exchange is an all-gather of the ranks' gradients
        for step in range(2):
            g = src.grads(step)
            local = g[w0 * Tu:(w0 + nl) * Tu]
            flat = torch.cat([t.reshape(-1) for t in local])
            out = torch.empty(world * flat.numel(), dtype=flat.dtype)
            transport.all_gather_flat(out, flat)
            gathered = list(torch.split(out, list(numel) * n))
            for a, b in zip(gathered, g):
                assert torch.equal(a, b)  # every worker's gradient, in [worker][tensor] order
            ref.warmup_step([W.to_numpy_grad(t) for t in g])
            mine.warmup_step([W.to_numpy_grad(t) for t in gathered])
        ref.freeze()
        mine.freeze()
        x, m, den = mine.view("x").copy(), mine.view("m").copy(), mine.view("den").copy()
        delta = np.zeros((n, D_), np.float32)
        eps = np.zeros(D_, np.float32)
        wbits = np.zeros((n, Wd), np.uint32)
        wscale = np.zeros((n, T), np.float32)
        sbits = np.zeros((1, Wd), np.uint32)
        sscale = np.zeros((T, n), np.float32)
        regions = [wbits, wscale.view(np.uint32), sbits, sscale.view(np.uint32)]
        b1 = np.float32(w.beta1)
        omb1 = np.float32(1.0) - b1
        nf = np.float32(n)
        for step in range(2, 5):
            g = src.grads(step)
            ref.compress_step([W.to_numpy_grad(t) for t in g])
            # ---- begin: this rank's workers
            for il in range(nl):
                i = w0 + il
                gi = np.concatenate([_decode(t).reshape(-1) for t in g[i * Tu:(i + 1) * Tu]]) if D_ else np.zeros(0, np.float32)
                cv = (b1 * m + omb1 * gi) + delta[i]
                for k, L in enumerate(segs):
                    s, words, err = oracle.compress(cv[soff[k]:soff[k + 1]])
                    wscale[i, k] = s
                    wbits[i, woff[k]:woff[k + 1]] = words
                    delta[i, soff[k]:soff[k + 1]] = err
            send = np.zeros((world, send_block), np.uint32)
            _apply(rows, 0, regions, send)
            recv_t = torch.zeros(world * send_block, dtype=torch.int32)
            transport.all_to_all(recv_t, torch.from_numpy(send.view(np.int32).reshape(-1).copy()))
            recv = recv_t.numpy().view(np.uint32).reshape(world, send_block).copy()
            # ---- serve: unpack, then this rank's shards
            _apply(rows, 1, regions, recv)
            for k, L in enumerate(segs):
                if L == 0:
                    continue
                bits = [_bits(wbits[i, woff[k]:woff[k + 1]], L) for i in range(n)]
                for j in range(w0, w0 + nl):
                    lo, hi = oracle.shard(L, n, j)
                    if hi <= lo:
                        continue
                    acc = np.zeros(hi - lo, np.float32)
                    for i in range(n):
                        s = wscale[i, k]
                        acc = acc + np.where(bits[i][lo:hi], s, -s).astype(np.float32)
                    a = acc / nf + eps[soff[k] + lo: soff[k] + hi]
                    S, words, err = oracle.compress(a)
                    sscale[k, j] = S
                    sbits[0, woff[k] + lo // 32: woff[k] + lo // 32 + len(words)] = words
                    eps[soff[k] + lo: soff[k] + hi] = err
            bcast = np.zeros((1, bcast_block), np.uint32)
            _apply(rows, 2, regions, bcast)
            gath_t = torch.zeros(world * bcast_block, dtype=torch.int32)
            transport.all_gather(gath_t, torch.from_numpy(bcast.view(np.int32).reshape(-1).copy()))
            gath = gath_t.numpy().view(np.uint32).reshape(world, bcast_block).copy()
            # ---- end: the broadcast momentum and the update
            _apply(rows, 3, regions, gath)
            for k, L in enumerate(segs):
                if L == 0:
                    continue
                sb = _bits(sbits[0, woff[k]:woff[k + 1]], L)
                for j in range(n):
                    lo, hi = oracle.shard(L, n, j)
                    S = sscale[k, j]
                    m[soff[k] + lo: soff[k] + hi] = np.where(sb[lo:hi], S, -S)
            x = x - np.float32(w.lr) * (m / den)
            # ---- every rank agrees with the single-process oracle, bit for bit
            assert np.array_equal(sbits[0], ref.view("sbits")), (rank, step, "server words")
            assert np.array_equal(sscale.view(np.uint32), ref.sscale.view(np.uint32)), (rank, step, "server scales")
            assert np.array_equal(wscale.view(np.uint32), ref.wscale.view(np.uint32)), (rank, step, "worker scales")
            assert np.array_equal(m.view(np.uint32), ref.view("m").view(np.uint32)), (rank, step, "m")
            assert np.array_equal(x.view(np.uint32), ref.view("x").view(np.uint32)), (rank, step, "x")
            for il in range(nl):
                i = w0 + il
                assert np.array_equal(wbits[i], ref.view("wbits")[i]), (rank, step, i)
                assert np.array_equal(delta[i].view(np.uint32), ref.view("delta")[i].view(np.uint32)), (rank, step, i)
            for k, L in enumerate(segs):  # other ranks' workers: their words of this rank's shards
                for j in range(w0, w0 + nl):
                    lo, hi = oracle.shard(L, n, j)
                    if hi > lo:
                        a0, a1 = woff[k] + lo // 32, woff[k] + (hi + 31) // 32
                        for i in range(n):
                            assert np.array_equal(wbits[i, a0:a1], ref.view("wbits")[i, a0:a1]), (rank, step, k, j, i)
                        e = slice(soff[k] + lo, soff[k] + hi)
                        assert np.array_equal(eps[e].view(np.uint32), ref.view("eps_srv")[e].view(np.uint32))
    finally:
        tdist.destroy_process_group()


@pytest.mark.parametrize("case", list(CASES))
def test_two_cpu_ranks_match_one_process(case):
    import torch.multiprocessing as mp

    mp.spawn(_rank_main, args=(CASES[case]["world"], _free_port(), case), nprocs=CASES[case]["world"], join=True)
