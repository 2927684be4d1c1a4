"""ORACLE for the 1-bit Adam optimizer step -- TEST INFRASTRUCTURE ONLY.

Plain single-threaded C (``onebit_oracle.c``) behind a thin ctypes binding.  Only the test suite,
the package's ``smoke()`` check and the benchmark's CPU-baseline / reference leg may import this
module.  It shares nothing with the CUDA library: no code, header, table or constant.  Sources and
the precision reading are stated in ``onebit_oracle.h``.

Every function follows "1-bit Adam: Communication Efficient Large-Scale Training with Adam's
Convergence Speed" (Tang et al.): Sec. 4.3 (sign + magnitude-preserving scale), Sec. 11 (worker
error-compensated compression, server average + recompression, broadcast) and the summary formulas of
the AIMech page "1-bit Adam (Two-Stage Preconditioner-Frozen Error-Compensated Adam)".

Parity pins for every function are in ``tests/test_oracle_pins.py``; none is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "onebit_oracle.c")
_LIB = os.path.join(_HERE, "libonebit_oracle.so")

F32, F16, BF16 = 0, 1, 2
_f32p = ctypes.POINTER(ctypes.c_float)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_i64p = ctypes.POINTER(ctypes.c_int64)


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("beta1", ctypes.c_float),
        ("beta2", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("lr", ctypes.c_float),
        ("n_workers", ctypes.c_int32),
        ("n_tensors", ctypes.c_int32),
        ("numel", _i64p),
        ("grad_dtype", ctypes.c_int32),
        ("bias_correction", ctypes.c_int32),
    ]


def build(force: bool = False, src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile the oracle with gcc (-O2, no floating-point contraction)."""
    hdr = os.path.join(_HERE, "onebit_oracle.h")
    if force or not os.path.exists(out) or os.path.getmtime(out) < max(os.path.getmtime(src),
                                                                        os.path.getmtime(hdr)):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
             "-I", _HERE, *extra_flags, "-o", tmp, src, "-lm"]
        )
        os.replace(tmp, out)
    return out


class OracleLib:
    """ctypes view of one build of the oracle library (the default build, or a test's copy)."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        L.ora_half_to_float.restype = ctypes.c_float
        L.ora_half_to_float.argtypes = [ctypes.c_uint16]
        L.ora_bf16_to_float.restype = ctypes.c_float
        L.ora_bf16_to_float.argtypes = [ctypes.c_uint16]
        L.ora_words.restype = ctypes.c_int64
        L.ora_words.argtypes = [ctypes.c_int64]
        L.ora_shard.restype = None
        L.ora_shard.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _i64p, _i64p]
        L.ora_rms.restype = ctypes.c_float
        L.ora_rms.argtypes = [_f32p, ctypes.c_int64]
        L.ora_norm2.restype = ctypes.c_double
        L.ora_norm2.argtypes = [_f32p, ctypes.c_int64]
        L.ora_pack_signs.restype = None
        L.ora_pack_signs.argtypes = [_f32p, ctypes.c_int64, _u32p]
        L.ora_unpack_signs.restype = None
        L.ora_unpack_signs.argtypes = [_u32p, ctypes.c_int64, ctypes.c_float, _f32p]
        L.ora_compress.restype = ctypes.c_float
        L.ora_compress.argtypes = [_f32p, ctypes.c_int64, _u32p, _f32p]
        vpp = ctypes.POINTER(ctypes.c_void_p)
        L.ora_warmup_step.restype = ctypes.c_int
        L.ora_warmup_step.argtypes = [ctypes.POINTER(_Cfg), ctypes.c_int64, _f32p, _f32p, _f32p, vpp]
        L.ora_freeze.restype = ctypes.c_int
        L.ora_freeze.argtypes = [ctypes.POINTER(_Cfg), ctypes.c_int64, _f32p, _f32p]
        L.ora_compress_step.restype = ctypes.c_int
        L.ora_compress_step.argtypes = [ctypes.POINTER(_Cfg), _f32p, _f32p, _f32p, _f32p, _f32p, vpp,
                                        _u32p, _f32p, _u32p, _f32p]
        L.ora_ec_adam_step.restype = ctypes.c_int
        L.ora_ec_adam_step.argtypes = [ctypes.POINTER(_Cfg), ctypes.c_int64, _f32p, _f32p, _f32p, _f32p, _f32p,
                                       vpp, _u32p, _f32p, _u32p, _f32p]
        self.c = L
        self.path = path

    # ------------------------------------------------------------ element helpers
    def half_to_float(self, h: int) -> float:
        return self.c.ora_half_to_float(int(h) & 0xFFFF)

    def bf16_to_float(self, b: int) -> float:
        return self.c.ora_bf16_to_float(int(b) & 0xFFFF)

    def words(self, n: int) -> int:
        return int(self.c.ora_words(int(n)))

    def shard(self, length: int, n: int, j: int) -> tuple[int, int]:
        lo, hi = ctypes.c_int64(), ctypes.c_int64()
        self.c.ora_shard(int(length), int(n), int(j), ctypes.byref(lo), ctypes.byref(hi))
        return lo.value, hi.value

    def rms(self, v: np.ndarray) -> np.float32:
        v = np.ascontiguousarray(v, dtype=np.float32)
        return np.float32(self.c.ora_rms(_fp(v), v.size))

    def norm2(self, v: np.ndarray) -> float:
        v = np.ascontiguousarray(v, dtype=np.float32)
        if v.size == 0:
            return 0.0
        return float(self.c.ora_norm2(_fp(v), v.size))

    def pack_signs(self, v: np.ndarray) -> np.ndarray:
        v = np.ascontiguousarray(v, dtype=np.float32)
        out = np.zeros(max(self.words(v.size), 1), dtype=np.uint32)
        self.c.ora_pack_signs(_fp(v), v.size, _up(out))
        return out[: self.words(v.size)]

    def unpack_signs(self, w: np.ndarray, length: int, scale: float) -> np.ndarray:
        w = np.ascontiguousarray(w, dtype=np.uint32)
        if w.size == 0:
            w = np.zeros(1, np.uint32)
        out = np.zeros(max(length, 1), dtype=np.float32)
        self.c.ora_unpack_signs(_up(w), int(length), float(scale), _fp(out))
        return out[:length]

    def compress(self, c: np.ndarray) -> tuple[np.float32, np.ndarray, np.ndarray]:
        """Returns (scale, sign words, error c - scale*sign(c))."""
        c = np.ascontiguousarray(c, dtype=np.float32)
        w = np.zeros(max(self.words(c.size), 1), dtype=np.uint32)
        err = np.zeros(max(c.size, 1), dtype=np.float32)
        cc = c if c.size else np.zeros(1, np.float32)
        s = self.c.ora_compress(_fp(cc), c.size, _up(w), _fp(err))
        return np.float32(s), w[: self.words(c.size)], err[: c.size]

    def optimizer(self, *args, **kw) -> "OneBitAdamOracle":
        return OneBitAdamOracle(*args, lib=self, **kw)


_default = None


def lib() -> OracleLib:
    global _default
    if _default is None:
        _default = OracleLib(build())
    return _default


def _fp(a: np.ndarray):
    assert a.dtype == np.float32 and a.flags.c_contiguous
    return a.ctypes.data_as(_f32p)


def _up(a: np.ndarray):
    assert a.dtype == np.uint32 and a.flags.c_contiguous
    return a.ctypes.data_as(_u32p)


def half_to_float(h):
    return lib().half_to_float(h)


def bf16_to_float(b):
    return lib().bf16_to_float(b)


def words(n):
    return lib().words(n)


def shard(length, n, j):
    return lib().shard(length, n, j)


def rms(v):
    return lib().rms(v)


def norm2(v):
    return lib().norm2(v)


def pack_signs(v):
    return lib().pack_signs(v)


def unpack_signs(w, length, scale):
    return lib().unpack_signs(w, length, scale)


def compress(c):
    return lib().compress(c)


# ---------------------------------------------------------------- the optimizer

def scale_blocks(numel, block):
    """Sizes of the compressed segments: the tensors themselves (block 0), or each tensor cut into
    consecutive blocks of ``block`` elements, the last one shorter, an empty tensor one empty block."""
    if not block:
        return [int(v) for v in numel]
    out = []
    for L in numel:
        L = int(L)
        out.extend([min(block, L - s) for s in range(0, L, block)] if L else [0])
    return out


class OneBitAdamOracle:
    """Whole optimizer state on the host, stepped by the C oracle.

    ``numel``: list of tensor sizes (one entry = one flat buffer).  Per-element arrays are the
    concatenation of the tensors.  Gradients are passed per step as a list of n*T numpy arrays
    ordered [worker][tensor]: float32 arrays, float16 arrays, or uint16 arrays of bfloat16 bits.

    ``scale_block`` B > 0 is the per-chunk parameter-server form ("1-bit Adam ...", Sec. 11: the
    server role is taken per chunk): every tensor is cut into consecutive blocks of B elements (the
    last one shorter; an empty tensor stays one empty block) and each block is compressed as a tensor
    of its own.  ``numel``, ``T`` and the scale arrays then describe the blocks; gradients are still
    passed per caller tensor (``unumel``).
    """

    def __init__(self, numel, n_workers, x0, beta1=0.9, beta2=0.999, eps=1e-8, lr=1e-3,
                 grad_dtype=F32, bias_correction=False, lib: OracleLib | None = None, scale_block=0):
        self.lib = lib if lib is not None else globals()["lib"]()
        self.unumel = [int(v) for v in numel]
        self.scale_block = int(scale_block)
        self.numel = scale_blocks(self.unumel, self.scale_block)
        self.n = int(n_workers)
        self.T = len(self.numel)
        self.D = sum(self.numel)
        self.W = sum(self.lib.words(v) for v in self.numel)
        self._numel_arr = (ctypes.c_int64 * self.T)(*self.numel)
        self.cfg = _Cfg(beta1, beta2, eps, lr, self.n, self.T,
                        ctypes.cast(self._numel_arr, _i64p), grad_dtype, int(bias_correction))
        self.grad_dtype = grad_dtype
        D1 = max(self.D, 1)
        self.x = np.ascontiguousarray(np.asarray(x0, dtype=np.float32).reshape(-1)).copy()
        assert self.x.size == self.D
        if self.x.size == 0:
            self.x = np.zeros(1, np.float32)
        self.m = np.zeros(D1, np.float32)
        self.v = np.zeros(D1, np.float32)
        self.den = np.zeros(D1, np.float32)
        self.delta = np.zeros((self.n, D1), np.float32)
        self.eps_srv = np.zeros(D1, np.float32)
        self.wbits = np.zeros((self.n, max(self.W, 1)), np.uint32)
        self.wscale = np.zeros((self.n, self.T), np.float32)
        self.sbits = np.zeros(max(self.W, 1), np.uint32)
        self.sscale = np.zeros((self.T, self.n), np.float32)
        self.t = 0
        self.phase = "warmup"

    def set_lr(self, lr):
        """Learning rate of the following steps (the method keeps it fixed; schedules change it)."""
        self.cfg.lr = float(lr)

    def _grad_ptrs(self, grads):
        if self.scale_block:  # cut each caller tensor's gradient into its blocks
            Tu, B = len(self.unumel), self.scale_block
            assert len(grads) == self.n * Tu
            cut = []
            for i in range(self.n):
                for k, L in enumerate(self.unumel):
                    g = np.ascontiguousarray(grads[i * Tu + k])
                    cut.extend([g[s: s + B] for s in range(0, L, B)] if L else [g])
            grads = cut
        assert len(grads) == self.n * self.T
        keep = []
        ptrs = (ctypes.c_void_p * len(grads))()
        for idx, g in enumerate(grads):
            g = np.ascontiguousarray(g)
            k = idx % self.T
            assert g.size == self.numel[k], (g.size, self.numel[k])
            if self.grad_dtype == F32:
                assert g.dtype == np.float32
            else:
                assert g.dtype in (np.float16, np.uint16, np.int16)
            keep.append(g)
            ptrs[idx] = g.ctypes.data if g.size else None
        return ptrs, keep

    def warmup_step(self, grads):
        assert self.phase == "warmup"
        self.t += 1
        ptrs, keep = self._grad_ptrs(grads)
        rc = self.lib.c.ora_warmup_step(ctypes.byref(self.cfg), self.t, _fp(self.x), _fp(self.m), _fp(self.v), ptrs)
        assert rc == 0

    def freeze(self):
        assert self.phase == "warmup" and self.t >= 1
        rc = self.lib.c.ora_freeze(ctypes.byref(self.cfg), self.t, _fp(self.v), _fp(self.den))
        assert rc == 0
        self.delta[:] = 0
        self.eps_srv[:] = 0
        self.phase = "compress"

    def compress_step(self, grads):
        assert self.phase == "compress"
        self.t += 1
        ptrs, keep = self._grad_ptrs(grads)
        rc = self.lib.c.ora_compress_step(ctypes.byref(self.cfg), _fp(self.x), _fp(self.m), _fp(self.den),
                                     _fp(self.delta), _fp(self.eps_srv), ptrs, _up(self.wbits),
                                     _fp(self.wscale), _up(self.sbits), _fp(self.sscale))
        assert rc == 0

    def ec_adam_step(self, grads):
        """The baseline of error-compensated 1-bit compression applied to the gradients, then Adam
        ("1-bit Adam ...", Sec. 3.2).  Legal in the warm-up phase; shares m, v and the error memories."""
        assert self.phase == "warmup"
        self.t += 1
        ptrs, keep = self._grad_ptrs(grads)
        rc = self.lib.c.ora_ec_adam_step(ctypes.byref(self.cfg), self.t, _fp(self.x), _fp(self.m), _fp(self.v),
                                         _fp(self.delta), _fp(self.eps_srv), ptrs, _up(self.wbits),
                                         _fp(self.wscale), _up(self.sbits), _fp(self.sscale))
        assert rc == 0

    # views without the size-1 placeholder used for empty lists
    def view(self, name):
        a = getattr(self, name)
        if name in ("x", "m", "v", "den", "eps_srv"):
            return a[: self.D]
        if name == "delta":
            return a[:, : self.D]
        if name == "wbits":
            return a[:, : self.W]
        if name == "sbits":
            return a[: self.W]
        return a
