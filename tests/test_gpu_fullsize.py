"""Full-size workloads in the benchmark's launch configuration.

At these sizes the oracle cannot run the whole problem, so two kinds of checks are made:

* sampled outputs the oracle computes one coordinate at a time: the warm-up Adam steps and the
  freeze are elementwise, and the first compression step's sign bits depend only on the coordinate's
  own momentum and gradients.  The oracle runs on the sampled coordinates alone (a few thousand:
  random ones plus shard boundaries and tensor ends) with the same seeded gradients, and x, m, v, den
  and the worker sign bits must match bit for bit;
* properties that hold at any size, checked in fp64 on the GPU's complete exported state, streamed
  over slices: scale * sqrt(L) = ||c||_2 for every worker and tensor (c rebuilt as error +
  scale*sign), c = b1*m + (1-b1)*g + previous error, bits = [c >= 0], the server input equals the
  average of the decompressed worker messages plus the previous server error, S * sqrt(len) = ||a||_2
  per shard, the broadcast m = S*sign(a), and the update x' = x - lr*m/den.
"""
import math

import numpy as np
import pytest
import torch

import communication_compressed_optimizer_compress_gb300 as ob
import oracle
from communication_compressed_optimizer_compress_gb300 import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SLICE = 1 << 25


def _samples(w, n_random=4096, seed=123):
    rng = np.random.default_rng(seed)
    pts = set(rng.integers(0, w.d, n_random).tolist())
    off = 0
    for k, L in enumerate(w.numel):
        if k < 40 or k == len(w.numel) - 1:
            for j in range(w.n_workers):
                lo, hi = oracle.shard(L, w.n_workers, j)
                for e in (lo, lo + 1, hi - 1, hi - 2):
                    if lo <= e < hi:
                        pts.add(off + e)
            for e in (0, L - 1, L - 8, L - 9, L - 33):
                if 0 <= e < L:
                    pts.add(off + e)
        off += L
    return np.array(sorted(pts), dtype=np.int64)


def _flat(tensors):
    return tensors[0].reshape(-1) if len(tensors) == 1 else torch.cat([t.reshape(-1) for t in tensors])


def _bits_flat(words, numel):
    """Sign words in the tensor-wise layout -> uint8 0/1 per element of the concatenation."""
    w = words.view(torch.int32)
    bits = ((w.unsqueeze(1) >> torch.arange(32, device=w.device, dtype=torch.int32)) & 1).to(torch.uint8).reshape(-1)
    if len(numel) == 1:
        return bits[: numel[0]]
    parts, woff = [], 0
    for L in numel:
        parts.append(bits[woff * 32: woff * 32 + L])
        woff += (L + 31) // 32
    return torch.cat(parts)


def _run(name, compress_steps=2):
    w = W.WORKLOADS[name]
    dev = torch.device("cuda:0")
    n, numel, D, T = w.n_workers, list(w.numel), w.d, w.n_tensors
    E = _samples(w)
    E_dev = torch.from_numpy(E).to(dev)
    offs = np.concatenate([[0], np.cumsum(numel)]).astype(np.int64)
    per_shard = [32 * -(-L // (32 * n)) for L in numel]

    params = W.params(w, dev)
    opt = ob.OneBitAdam(params, n, w.warmup_steps, w.beta1, w.beta2, w.eps, w.lr,
                        grad_dtype=W.TORCH_DTYPE[w.grad_dtype])
    ora = oracle.OneBitAdamOracle([len(E)], n, _flat(params)[E_dev].cpu().numpy(), w.beta1, w.beta2, w.eps, w.lr,
                                  grad_dtype=w.grad_dtype)
    src = W.GradSource(w, dev)

    def grads(step):
        g = src.grads(step)
        gs = [W.to_numpy_grad(_flat(g[i * T:(i + 1) * T])[E_dev]) for i in range(n)]
        return g, gs

    # ---- warm-up Adam and freeze: elementwise, sampled, bit-exact
    step = 0
    for _ in range(w.warmup_steps):
        g, gs = grads(step)
        step += 1
        opt.warmup_step(g)
        ora.warmup_step(gs)
        del g
    torch.cuda.synchronize()
    for got, want in ((_flat(params)[E_dev], ora.view("x")), (opt.export_state(ob.STATE_M)[E_dev], ora.view("m")),
                      (opt.export_state(ob.STATE_V)[E_dev], ora.view("v"))):
        assert np.array_equal(got.cpu().numpy().view(np.uint32), want.view(np.uint32))
    opt.freeze_variance()
    ora.freeze()
    den = opt.export_state(ob.STATE_V)
    assert np.array_equal(den[E_dev].cpu().numpy().view(np.uint32), ora.view("den").view(np.uint32))

    b1 = torch.tensor(np.float32(w.beta1), device=dev)
    omb1 = torch.tensor(np.float32(1.0) - np.float32(w.beta1), device=dev)
    lr = torch.tensor(np.float32(w.lr), device=dev)
    err_prev = [torch.zeros(D, device=dev) for _ in range(n)]
    eps_prev = torch.zeros(D, device=dev)
    seg_starts = torch.from_numpy(offs[1:]).to(dev)
    per_dev = torch.tensor(per_shard, device=dev, dtype=torch.int64)
    offs_dev = torch.from_numpy(offs).to(dev)
    for cstep in range(compress_steps):
        m_prev = opt.export_state(ob.STATE_M)
        x_prev = _flat(params).clone()
        g, gs = grads(step)
        step += 1
        opt.compress_step(g)
        if cstep == 0:
            ora.compress_step(gs)
        torch.cuda.synchronize()
        assert opt.get_status() == ob.OK
        ws = opt.export_state(ob.STATE_WORKER_SCALES).reshape(n, T).double()
        ss = opt.export_state(ob.STATE_SERVER_SCALES).reshape(T, n).double()
        errs = [opt.export_state(ob.STATE_WORKER_ERROR, i) for i in range(n)]
        bits = [_bits_flat(opt.export_state(ob.STATE_WORKER_BITS, i), numel) for i in range(n)]
        sbits = _bits_flat(opt.export_state(ob.STATE_SERVER_BITS), numel)
        eps_now = opt.export_state(ob.STATE_SERVER_ERROR)
        m_now = opt.export_state(ob.STATE_M)
        x_now = _flat(params)
        gflat = [_flat(g[i * T:(i + 1) * T]) for i in range(n)]
        if cstep == 0:  # sampled worker bits against the oracle
            for i in range(n):
                ob_bits = ((torch.from_numpy(ora.view("wbits")[i].view(np.int32).copy()).to(dev).unsqueeze(1)
                            >> torch.arange(32, device=dev, dtype=torch.int32)) & 1).reshape(-1)[: len(E)]
                assert torch.equal(bits[i][E_dev].to(torch.int32), ob_bits), i
        w_sumsq = torch.zeros(n, T, device=dev, dtype=torch.float64)
        s_sumsq = torch.zeros(T * n, device=dev, dtype=torch.float64)
        for lo in range(0, D, SLICE):
            hi = min(D, lo + SLICE)
            idx = torch.arange(lo, hi, device=dev)
            seg = torch.bucketize(idx, seg_starts, right=True)
            shard = (idx - offs_dev[seg]) // per_dev[seg]
            avg = torch.zeros(hi - lo, device=dev, dtype=torch.float64)
            for i in range(n):
                s_el = ws[i][seg]
                sgn = torch.where(bits[i][lo:hi].bool(), s_el, -s_el)
                c = errs[i][lo:hi].double() + sgn
                w_sumsq[i].index_add_(0, seg, c * c)
                c32 = (b1 * m_prev[lo:hi] + omb1 * gflat[i][lo:hi].float()) + err_prev[i][lo:hi]
                tol = 1e-7 + 1e-5 * c32.double().abs() + 2e-7 * s_el
                assert bool(((c - c32.double()).abs() <= tol).all()), (name, cstep, i, lo)
                near0 = c32.double().abs() < 1e-7 * s_el
                assert bool(((bits[i][lo:hi] == (c32 >= 0).to(torch.uint8)) | near0).all()), (name, cstep, i, lo)
                avg += sgn
            avg /= n
            S_el = ss[seg, shard]
            a = eps_now[lo:hi].double() + torch.where(sbits[lo:hi].bool(), S_el, -S_el)
            want_a = avg + eps_prev[lo:hi].double()
            assert bool(((a - want_a).abs() <= 1e-7 + 1e-5 * want_a.abs() + 2e-7 * S_el).all()), (name, cstep, lo)
            s_sumsq.index_add_(0, seg * n + shard, a * a)
            assert torch.equal(m_now[lo:hi].double(), torch.where(sbits[lo:hi].bool(), S_el, -S_el))
            x_want = x_prev[lo:hi] - lr * (m_now[lo:hi] / den[lo:hi])
            assert bool(((x_now[lo:hi] - x_want).abs() <= 1e-7 + 1e-6 * x_want.abs()).all()), (name, cstep, lo)
        L64 = torch.tensor(numel, device=dev, dtype=torch.float64)
        got = ws * torch.sqrt(L64)
        ref = torch.sqrt(w_sumsq)
        assert bool(((got - ref).abs() <= 2e-6 * ref).all()), (name, cstep, (got - ref).abs().max())
        lens = torch.tensor([[oracle.shard(L, n, j)[1] - oracle.shard(L, n, j)[0] for j in range(n)] for L in numel],
                            device=dev, dtype=torch.float64).reshape(-1)
        got = ss.reshape(-1) * torch.sqrt(lens)
        ref = torch.sqrt(s_sumsq)
        assert bool(((got - ref).abs() <= 2e-6 * ref).all()), (name, cstep, (got - ref).abs().max())
        err_prev, eps_prev = errs, eps_now
        del g, gflat, bits
    opt.free()
    del err_prev, eps_prev
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["bert_large", "bert_base", "ragged_bert_large", "gpt2_1p5b", "over_2g"])
def test_full_size(name):
    _run(name)
