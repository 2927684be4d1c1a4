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
    with np.errstate(invalid="ignore"):
        bad = ~((got == want) | (np.abs(got - want) <= atol + rtol * np.abs(want)))  # equal infinities pass
    bad |= np.isnan(got) != np.isnan(want)
    if bad.any():
        idx = np.flatnonzero(bad)[:5]
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} differ, e.g. at {idx}: "
                             f"gpu {got[idx]} oracle {want[idx]}")


def _close_t(name, got, want, mask=None, rtol=RTOL, atol=ATOL):
    """_close on device tensors (fp64); rtol may be a tensor of the same shape as got."""
    got = got.reshape(-1).double()
    want = want.reshape(-1).double().to(got.device)
    if torch.is_tensor(rtol):
        rtol = rtol.reshape(-1).to(got.device)
    if mask is not None:
        got, want = got[mask], want[mask]
        if torch.is_tensor(rtol):
            rtol = rtol[mask]
    bad = ~((got == want) | ((got - want).abs() <= atol + rtol * want.abs()))  # equal infinities pass
    bad |= torch.isnan(got) != torch.isnan(want)
    if bool(bad.any()):
        idx = torch.nonzero(bad)[:5].flatten()
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.numel()} differ, e.g. at {idx.tolist()}: "
                             f"gpu {got[idx].tolist()} oracle {want[idx].tolist()}")


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

    def __init__(self, w: W.Workload, device="cuda:0", bias_correction=False, misalign=False, scale_block=0,
                 gen_device="cpu"):
        self.w = w
        self.dev = torch.device(device)
        # the seeded inputs are drawn on `gen_device` (the device is faster for the large cases); both
        # sides get the same values: the CUDA path the tensors, the oracle their host copies
        self.src = W.GradSource(w, gen_device)
        x0 = [p.cpu() for p in W.params(w, gen_device)]
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

    def _index(self):
        """Element -> (sign word, bit, segment, server shard) tables on the device, built once."""
        if getattr(self, "_idx", None) is None:
            dev, n = self.dev, self.w.n_workers
            D, T = self.D, len(self.numel)
            word = torch.empty(D, dtype=torch.int64, device=dev)
            bit = torch.empty(D, dtype=torch.int32, device=dev)
            seg = torch.empty(D, dtype=torch.int64, device=dev)
            shard = torch.empty(D, dtype=torch.int64, device=dev)
            for k, L in enumerate(self.numel):
                if L == 0:
                    continue
                a, b = int(self.offs[k]), int(self.offs[k + 1])
                e = torch.arange(L, device=dev, dtype=torch.int64)
                word[a:b] = int(self.woffs[k]) + e // 32
                bit[a:b] = (e % 32).to(torch.int32)
                seg[a:b] = k
                per = 32 * -(-L // (32 * n))
                shard[a:b] = k * n + e // per
            self._idx = (word, bit, seg, shard)
        return self._idx

    def _unpack(self, words):
        """Sign words (tensor-wise word layout, any 32-bit dtype) -> bool per element, on the device."""
        word, bit, _, _ = self._index()
        if not torch.is_tensor(words):
            words = torch.from_numpy(np.ascontiguousarray(words).view(np.int32))
        w = words.to(self.dev).view(torch.int32)
        return ((w[word] >> bit) & 1).bool()

    def _dev(self, a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)

    def check_compress(self, ec=False):
        """The parity protocol (module docstring), evaluated in fp64 on the device."""
        torch.cuda.synchronize()
        assert self.gpu.get_status() == ob.OK
        o, n, dev = self.ora, self.w.n_workers, self.dev
        T = len(self.numel)
        st = self.stats
        st.steps += 1
        st.coords += self.D
        _, _, seg, shard = self._index()
        numel_t = torch.tensor(self.numel, dtype=torch.float64, device=dev)
        gws = self.gpu.export_state(ob.STATE_WORKER_SCALES).reshape(n, T).double()
        gss = self.gpu.export_state(ob.STATE_SERVER_SCALES).reshape(T, n).double()
        ows = self._dev(o.wscale).reshape(n, T).double()
        oss = self._dev(o.sscale).reshape(T, n).double()
        # Coordinates excluded at an earlier step stay excluded everywhere: once the two sides
        # carry different error memories or a different m there, every later value at that
        # coordinate may differ.
        G = self._dev(self.excl_s)
        band_any = torch.zeros(self.D, dtype=torch.bool, device=dev)
        n_band_w = 0
        # ---- workers
        for i in range(n):
            ob_bits = self._unpack(o.view("wbits")[i])
            s_el = ows[i][seg]
            d_ora = self._dev(o.view("delta")[i]).double()
            c_ora = d_ora + torch.where(ob_bits, s_el, -s_el)
            band = c_ora.abs() < BAND * s_el
            keep = ~(G | band)
            gw = self.gpu.export_state(ob.STATE_WORKER_BITS, i)
            g_bits = self._unpack(gw)
            bad = (g_bits != ob_bits) & keep
            if bool(bad.any()):
                raise AssertionError(f"worker {i}: sign bits differ at {torch.nonzero(bad)[:5].flatten().tolist()}")
            if bool(keep.all()):  # full words, padding bits included
                assert torch.equal(gw.view(torch.int32).cpu(), torch.from_numpy(
                    np.ascontiguousarray(o.view("wbits")[i]).view(np.int32)))
            gd = self.gpu.export_state(ob.STATE_WORKER_ERROR, i)
            _close_t(f"worker {i} error", gd, d_ora, keep)
            nex = torch.zeros(T, dtype=torch.float64, device=dev).index_add_(0, seg, (~keep).double())
            rt = 3e-7 + torch.where(numel_t > 0, 8.0 * nex / numel_t.clamp(min=1), torch.zeros_like(nex))
            _close_t(f"worker {i} scales", gws[i], ows[i], rtol=rt, atol=0.0)
            st.scales += T
            st.scales_exact += int((gws[i].float() == ows[i].float()).sum())
            band_any |= band
            n_band_w += int(band.sum())
        st.excluded_worker += n_band_w
        st.worker_draws += n * self.D
        # ---- server
        sb_ora = self._unpack(o.view("sbits"))
        S_el = oss.reshape(-1)[shard]
        e_ora = self._dev(o.view("eps_srv")).double()
        a_ora = e_ora + torch.where(sb_ora, S_el, -S_el)
        band_s = a_ora.abs() < BAND * S_el
        excl = G | band_any | band_s
        keep = ~excl
        gsb = self.gpu.export_state(ob.STATE_SERVER_BITS)
        g_sbits = self._unpack(gsb)
        bad = (g_sbits != sb_ora) & keep
        if bool(bad.any()):
            raise AssertionError(f"server sign bits differ at {torch.nonzero(bad)[:5].flatten().tolist()}")
        if bool(keep.all()):
            assert torch.equal(gsb.view(torch.int32).cpu(), torch.from_numpy(
                np.ascontiguousarray(o.view("sbits")).view(np.int32)))
        st.bit_words_compared += gsb.numel() * (n + 1)
        _close_t("server error", self.gpu.export_state(ob.STATE_SERVER_ERROR), e_ora, keep)
        _close_t("m", self.gpu.export_state(ob.STATE_M), self._dev(o.view("m")), keep)
        _close_t("x", self._x_dev(), self._dev(o.view("x")), keep)
        if ec:
            _close_t("v", self.gpu.export_state(ob.STATE_V), self._dev(o.view("v")), keep)
        lens = torch.tensor([oracle.shard(L, n, j)[1] - oracle.shard(L, n, j)[0]
                             for L in self.numel for j in range(n)], dtype=torch.float64, device=dev)
        nex = torch.zeros(T * n, dtype=torch.float64, device=dev).index_add_(0, shard, excl.double())
        rt = 3e-7 + torch.where(lens > 0, 8.0 * nex / lens.clamp(min=1), torch.zeros_like(nex))
        _close_t("server scales", gss.reshape(-1), oss.reshape(-1), rtol=rt, atol=0.0)
        st.scales += T * n
        st.scales_exact += int((gss.float() == oss.float()).sum())
        self.excl_s = excl.cpu().numpy()
        st.excluded_server = int(excl.sum())

    def _x_dev(self):
        if self.D == 0:
            return torch.zeros(0, device=self.dev)
        return torch.cat([p.detach().reshape(-1) for p in self.params])

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
