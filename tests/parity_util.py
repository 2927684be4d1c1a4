"""Free-running comparison of the CUDA path with the oracle on the same seeded inputs.

Both sides start from the same parameters and see the same gradients; nothing computed by the CUDA
path is ever fed to the oracle.  After every step the CUDA state is exported and compared:

* packed sign words: bit-exact, except coordinates where the oracle's value sits within
  1e-7 * scale of zero (|c| for a worker bit, |a| for a server bit), where a one-ulp difference in a
  scale can legitimately flip the sign.  Such a coordinate stays excluded for the rest of the run
  (for that worker, and for the server, m and x at that coordinate), because the two sides then
  carry different error memories there;
* fp32 state (x, m, v/den, worker errors, server error): |gpu - oracle| <= 1e-7 + 1e-5 |oracle|;
* scales: within 3e-7 relative (one ulp of the final fp32 rounding, plus slack), widened by the
  excluded coordinates' possible effect on the norm; the fraction of exactly equal scales is reported.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import communication_compressed_optimizer_compress_gb300 as ob
import oracle
from communication_compressed_optimizer_compress_gb300 import workloads as W

RTOL, ATOL = 1e-5, 1e-7
BAND = 1e-7


@dataclasses.dataclass
class Stats:
    steps: int = 0
    scales: int = 0
    scales_exact: int = 0
    excluded_worker: int = 0   # (worker, coordinate, step) triples inside the exclusion band
    worker_draws: int = 0      # (worker, coordinate, step) triples compared
    excluded_server: int = 0   # coordinates excluded (sticky) at the last step
    coords: int = 0
    bit_words_compared: int = 0


def _close(name, got, want, mask=None, rtol=RTOL, atol=ATOL):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    if mask is not None:
        got, want = got[mask], want[mask]
    bad = ~(np.abs(got - want) <= atol + rtol * np.abs(want))
    bad |= np.isnan(got) != np.isnan(want)
    if bad.any():
        idx = np.flatnonzero(bad)[:5]
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} differ, e.g. at {idx}: "
                             f"gpu {got[idx]} oracle {want[idx]}")


def _bits(words, D, offs, woffs, numel):
    """Unpack sign words (tensor-wise word layout) into a bool vector of the D elements."""
    words = np.asarray(words).view(np.uint32)
    out = np.zeros(D, bool)
    for k, L in enumerate(numel):
        if L == 0:
            continue
        w = words[woffs[k]: woffs[k + 1]]
        b = ((w[:, None] >> np.arange(32, dtype=np.uint32)[None, :]) & 1).astype(bool).reshape(-1)[:L]
        out[offs[k]: offs[k + 1]] = b
    return out


class Pair:
    """A CUDA optimizer and an oracle optimizer stepped in lock-free parallel on the same inputs."""

    def __init__(self, w: W.Workload, device="cuda:0", bias_correction=False, misalign=False, scale_block=0):
        self.w = w
        self.dev = torch.device(device)
        self.src = W.GradSource(w, "cpu")
        x0 = W.params(w, "cpu")
        self.misalign = misalign
        if misalign:
            # parameters that start 4 bytes into an allocation: the kernels must take the scalar path
            self._pbuf = [torch.zeros(p.numel() + 1, device=self.dev) for p in x0]
            self.params = [b[1:] for b in self._pbuf]
            for p, x in zip(self.params, x0):
                p.copy_(x.to(self.dev))
        else:
            self.params = [p.to(self.dev) for p in x0]
        gdt = W.TORCH_DTYPE[w.grad_dtype]
        self.gpu = ob.OneBitAdam(self.params, w.n_workers, w.warmup_steps, w.beta1, w.beta2, w.eps, w.lr,
                                 grad_dtype=gdt, bias_correction=bias_correction, scale_block=scale_block)
        x0_np = torch.cat(x0).numpy() if sum(w.numel) else np.zeros(0, np.float32)
        self.ora = oracle.OneBitAdamOracle(list(w.numel), w.n_workers, x0_np, w.beta1, w.beta2, w.eps, w.lr,
                                           grad_dtype=w.grad_dtype, bias_correction=bias_correction,
                                           scale_block=scale_block)
        self.numel = list(self.ora.numel)  # the compressed segments: tensors, or their scale blocks
        self.D = sum(self.numel)
        self.offs = np.concatenate([[0], np.cumsum(self.numel)]).astype(np.int64)
        self.woffs = np.concatenate([[0], np.cumsum([(L + 31) // 32 for L in self.numel])]).astype(np.int64)
        self.step_idx = 0
        self.excl_w = np.zeros((w.n_workers, self.D), bool)
        self.excl_s = np.zeros(self.D, bool)
        self.stats = Stats()

    def _to_dev(self, g):
        if not self.misalign:
            return [t.to(self.dev) for t in g]
        out = []
        for t in g:
            buf = torch.zeros(t.numel() + 1, dtype=t.dtype, device=self.dev)
            buf[1:].copy_(t.to(self.dev))
            out.append(buf[1:])
        return out

    def grads(self):
        g = self.src.grads(self.step_idx)
        self.step_idx += 1
        return g

    def warmup(self, check=True):
        g = self.grads()
        self.gpu.warmup_step(self._to_dev(g))
        self.ora.warmup_step([W.to_numpy_grad(t) for t in g])
        if check:
            self.check_warmup()

    def freeze(self, check=True):
        self.gpu.freeze_variance()
        self.ora.freeze()
        if check:
            torch.cuda.synchronize()
            _close("den", self.gpu.export_state(ob.STATE_V).cpu().numpy(), self.ora.view("den"))

    def compress(self, check=True):
        g = self.grads()
        self.gpu.compress_step(self._to_dev(g))
        self.ora.compress_step([W.to_numpy_grad(t) for t in g])
        if check:
            self.check_compress()

    def ec_adam(self, check=True):
        """One step of the gradient-compression baseline on both sides."""
        g = self.grads()
        self.gpu.ec_adam_step(self._to_dev(g))
        self.ora.ec_adam_step([W.to_numpy_grad(t) for t in g])
        if check:
            self.check_compress(ec=True)

    def x(self):
        if self.D == 0:
            return np.zeros(0, np.float32)
        return torch.cat([p.detach().float().cpu() for p in self.params]).numpy()

    def check_warmup(self, exact=False):
        torch.cuda.synchronize()
        assert self.gpu.get_status() == ob.OK
        gx = self.x()
        gm = self.gpu.export_state(ob.STATE_M).cpu().numpy()
        gv = self.gpu.export_state(ob.STATE_V).cpu().numpy()
        if exact:
            assert np.array_equal(gx.view(np.uint32), self.ora.view("x").view(np.uint32))
            assert np.array_equal(gm.view(np.uint32), self.ora.view("m").view(np.uint32))
            assert np.array_equal(gv.view(np.uint32), self.ora.view("v").view(np.uint32))
        _close("x (warm-up)", gx, self.ora.view("x"))
        _close("m (warm-up)", gm, self.ora.view("m"))
        _close("v (warm-up)", gv, self.ora.view("v"))

    def check_compress(self, ec=False):
        torch.cuda.synchronize()
        assert self.gpu.get_status() == ob.OK
        w, o, n = self.w, self.ora, self.w.n_workers
        st = self.stats
        st.steps += 1
        st.coords += self.D
        gws = self.gpu.export_state(ob.STATE_WORKER_SCALES).cpu().numpy().reshape(n, -1)
        gss = self.gpu.export_state(ob.STATE_SERVER_SCALES).cpu().numpy().reshape(-1, n)
        seg_of = np.repeat(np.arange(len(self.numel)), self.numel)
        # Coordinates excluded at an earlier step stay excluded everywhere: once the two sides
        # carry different error memories or a different m there, every later value at that
        # coordinate may differ.
        G = self.excl_s.copy()
        band_w = np.zeros((n, self.D), bool)
        # ---- workers
        for i in range(n):
            ob_bits = _bits(o.view("wbits")[i], self.D, self.offs, self.woffs, self.numel)
            s_el = o.wscale[i][seg_of].astype(np.float64) if self.D else np.zeros(0)
            c_ora = o.view("delta")[i].astype(np.float64) + np.where(ob_bits, s_el, -s_el)
            band_w[i] = np.abs(c_ora) < BAND * s_el
            keep = ~(G | band_w[i])
            gw = self.gpu.export_state(ob.STATE_WORKER_BITS, i).cpu().numpy()
            g_bits = _bits(gw, self.D, self.offs, self.woffs, self.numel)
            if not np.array_equal(g_bits[keep], ob_bits[keep]):
                bad = np.flatnonzero((g_bits != ob_bits) & keep)[:5]
                raise AssertionError(f"worker {i}: sign bits differ at {bad}")
            if keep.all():  # full words, padding bits included
                assert np.array_equal(gw.view(np.uint32), o.view("wbits")[i])
            gd = self.gpu.export_state(ob.STATE_WORKER_ERROR, i).cpu().numpy()
            _close(f"worker {i} error", gd, o.view("delta")[i], keep)
            for k, L in enumerate(self.numel):
                nex = int((~keep[self.offs[k]: self.offs[k + 1]]).sum())
                rt = 3e-7 + (8.0 * nex / L if L else 0.0)
                _close(f"worker {i} scale of tensor {k}", gws[i, k], o.wscale[i, k], rtol=rt, atol=0)
                st.scales += 1
                st.scales_exact += int(np.float32(gws[i, k]) == o.wscale[i, k])
        self.excl_w |= band_w
        st.excluded_worker += int(band_w.sum())
        st.worker_draws += n * self.D
        # ---- server
        sb_ora = _bits(o.view("sbits"), self.D, self.offs, self.woffs, self.numel)
        S_el = np.zeros(self.D)
        for k, L in enumerate(self.numel):
            for j in range(n):
                lo, hi = oracle.shard(L, n, j)
                S_el[self.offs[k] + lo: self.offs[k] + hi] = o.sscale[k, j]
        a_ora = o.view("eps_srv").astype(np.float64) + np.where(sb_ora, S_el, -S_el)
        band_s = np.abs(a_ora) < BAND * S_el
        self.excl_s = G | band_w.any(axis=0) | band_s
        keep = ~self.excl_s
        gsb = self.gpu.export_state(ob.STATE_SERVER_BITS).cpu().numpy()
        g_sbits = _bits(gsb, self.D, self.offs, self.woffs, self.numel)
        if not np.array_equal(g_sbits[keep], sb_ora[keep]):
            bad = np.flatnonzero((g_sbits != sb_ora) & keep)[:5]
            raise AssertionError(f"server sign bits differ at {bad}")
        if keep.all():
            assert np.array_equal(gsb.view(np.uint32), o.view("sbits"))
        st.bit_words_compared += gsb.size * (n + 1)
        _close("server error", self.gpu.export_state(ob.STATE_SERVER_ERROR).cpu().numpy(), o.view("eps_srv"), keep)
        _close("m", self.gpu.export_state(ob.STATE_M).cpu().numpy(), o.view("m"), keep)
        _close("x", self.x(), o.view("x"), keep)
        if ec:
            _close("v", self.gpu.export_state(ob.STATE_V).cpu().numpy(), o.view("v"), keep)
        for k, L in enumerate(self.numel):
            for j in range(n):
                lo, hi = oracle.shard(L, n, j)
                nex = int(self.excl_s[self.offs[k] + lo: self.offs[k] + hi].sum())
                rt = 3e-7 + (8.0 * nex / (hi - lo) if hi > lo else 0.0)
                _close(f"server scale ({k},{j})", gss[k, j], o.sscale[k, j], rtol=rt, atol=0)
                st.scales += 1
                st.scales_exact += int(np.float32(gss[k, j]) == o.sscale[k, j])
        st.excluded_server = int(self.excl_s.sum())

    def run(self, warm=None, comp=None):
        warm = self.w.warmup_steps if warm is None else warm
        comp = self.w.compress_steps if comp is None else comp
        for _ in range(warm):
            self.warmup()
        self.freeze()
        for _ in range(comp):
            self.compress()
        return self.stats

    def close(self):
        self.gpu.free()
