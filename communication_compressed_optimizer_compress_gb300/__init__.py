"""GB300-native 1-bit Adam optimizer step (data-parallel hot path, n workers simulated on one GPU;
``dist.RankOneBitAdam`` spreads them over several GPUs).

Thin Python binding over the C ABI in ``include/onebit_adam.h`` (``libonebit_adam.so``, built by
``_build.build()``).  Every step of the method runs in the library's CUDA kernels; this module only
marshals pointers, sizes and the current torch stream.  If the library is missing, every entry point
raises: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# ONEBIT_LIBRARY=checked selects the checked build (kernels check their units of work against their
# buffers and report, instead of touching, any that would leave them); it is built on request by
# _build.build(checked=True)
CHECKED = os.environ.get("ONEBIT_LIBRARY", "") == "checked"
LIB_PATH = os.path.join(_HERE, "libonebit_adam_checked.so" if CHECKED else "libonebit_adam.so")

(OK, ERR_INVALID_ARG, ERR_PHASE, ERR_CUDA, ERR_NOMEM, ERR_WORKSPACE, ERR_NONFINITE, ERR_UNSUPPORTED,
 ERR_BOUNDS) = range(9)
F32, F16, BF16 = 0, 1, 2
PHASE_WARMUP, PHASE_COMPRESS = 0, 1
(STATE_M, STATE_V, STATE_WORKER_ERROR, STATE_SERVER_ERROR, STATE_WORKER_BITS, STATE_SERVER_BITS,
 STATE_WORKER_SCALES, STATE_SERVER_SCALES) = range(8)
FAULT_NONE, FAULT_STALL_COPIES, FAULT_FAIL_ALLOC, FAULT_TIGHTEN_BOUNDS = 0, 1, 2, 3
KERNEL_NAMES = ["warmup", "freeze", "worker", "worker_scale", "server", "server_scale", "update", "export",
                "ec_update", "exchange"]
NUM_KERNELS = len(KERNEL_NAMES)


class OneBitError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {error_string(status)} (status {status})"
        if detail:
            msg += f": {detail}"
        super().__init__(msg)


class Config(ctypes.Structure):
    _fields_ = [
        ("beta1", ctypes.c_float),
        ("beta2", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("lr", ctypes.c_float),
        ("warmup_steps", ctypes.c_int64),
        ("n_workers", ctypes.c_int32),
        ("n_tensors", ctypes.c_int32),
        ("numel", ctypes.POINTER(ctypes.c_int64)),
        ("grad_dtype", ctypes.c_int32),
        ("bias_correction", ctypes.c_int32),
        ("scale_block", ctypes.c_int64),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library.  Raises if it has not been built (no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"CUDA library {LIB_PATH} is missing: build it with "
                + ("`python -c 'from communication_compressed_optimizer_compress_gb300 import _build; "
                   "_build.build(checked=True)'`" if CHECKED else
                   "`python -c 'import __graft_entry__ as g; g.build()'`"))
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        cfgp = ctypes.POINTER(Config)
        st = ctypes.c_int
        sig = {
            "onebit_adam_workspace_size": [cfgp, ctypes.POINTER(sz)],
            "onebit_adam_init": [cfgp, ctypes.POINTER(vp), vp, sz, vp, ctypes.POINTER(vp)],
            "onebit_adam_warmup_step": [vp, ctypes.POINTER(vp), vp],
            "onebit_adam_freeze_variance": [vp, vp],
            "onebit_adam_compress_step": [vp, ctypes.POINTER(vp), vp],
            "onebit_adam_ec_adam_step": [vp, ctypes.POINTER(vp), vp],
            "onebit_adam_warmup_step_host": [vp, ctypes.POINTER(vp), vp],
            "onebit_adam_compress_step_host": [vp, ctypes.POINTER(vp), vp],
            "onebit_adam_free": [vp],
            "onebit_adam_get_status": [vp, vp],
            "onebit_adam_clear_status": [vp, vp],
            "onebit_adam_get_step": [vp, ctypes.POINTER(i64), ctypes.POINTER(i32)],
            "onebit_adam_set_step": [vp, i64, i32, vp],
            "onebit_adam_state_size": [vp, i32, ctypes.POINTER(sz)],
            "onebit_adam_export": [vp, i32, i32, vp, vp],
            "onebit_adam_import": [vp, i32, i32, vp, vp],
            "onebit_adam_comm_bytes": [vp, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)],
            "onebit_adam_set_timing": [vp, i32],
            "onebit_adam_kernel_times": [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)],
            "onebit_adam_launch_count": [vp, ctypes.POINTER(i64)],
            "onebit_adam_plan_chunks": [cfgp, ctypes.POINTER(i64), i64, ctypes.POINTER(i64)],
            "onebit_adam_plan_worker_chunks": [cfgp, ctypes.POINTER(i64), i64, ctypes.POINTER(i64)],
            "onebit_adam_set_fault_injection": [vp, i32, i64],
            "onebit_adam_set_max_ctas": [vp, i32],
            "onebit_adam_set_lr": [vp, ctypes.c_float],
            "onebit_adam_set_variance_monitor": [vp, i32],
            "onebit_adam_variance_norm": [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)],
            "onebit_adam_set_auto_freeze": [vp, ctypes.c_double],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = st
        L.onebit_adam_error_string.argtypes = [st]
        L.onebit_adam_error_string.restype = ctypes.c_char_p
        L.onebit_adam_last_error.argtypes = [vp]
        L.onebit_adam_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def error_string(status: int) -> str:
    return lib().onebit_adam_error_string(int(status)).decode()


def _check(status: int, where: str, handle=None):
    if status != OK:
        detail = ""
        if handle:
            detail = lib().onebit_adam_last_error(handle).decode()
        elif where == "onebit_adam_init":  # a failed init leaves its message on the thread
            detail = lib().onebit_adam_last_error(None).decode()
        raise OneBitError(status, where, detail)


def make_config(numel, n_workers, warmup_steps=1, beta1=0.9, beta2=0.999, eps=1e-8, lr=1e-3,
                grad_dtype=F32, bias_correction=False, scale_block=0):
    arr = (ctypes.c_int64 * len(numel))(*[int(v) for v in numel])
    cfg = Config(beta1, beta2, eps, lr, int(warmup_steps), int(n_workers), len(numel),
                 ctypes.cast(arr, ctypes.POINTER(ctypes.c_int64)), int(grad_dtype), int(bool(bias_correction)),
                 int(scale_block))
    cfg._keep = arr
    return cfg


def workspace_size(cfg: Config) -> int:
    out = ctypes.c_size_t()
    _check(lib().onebit_adam_workspace_size(ctypes.byref(cfg), ctypes.byref(out)), "onebit_adam_workspace_size")
    return out.value


def plan_chunks(cfg: Config):
    """The launcher's chunk table: list of (tensor, shard, start, length, padded offset)."""
    count = ctypes.c_int64()
    _check(lib().onebit_adam_plan_chunks(ctypes.byref(cfg), None, 0, ctypes.byref(count)), "onebit_adam_plan_chunks")
    rows = (ctypes.c_int64 * (5 * max(count.value, 1)))()
    _check(lib().onebit_adam_plan_chunks(ctypes.byref(cfg), rows, count.value, ctypes.byref(count)),
           "onebit_adam_plan_chunks")
    return [tuple(rows[5 * q: 5 * q + 5]) for q in range(count.value)]


def plan_worker_chunks(cfg: Config):
    """The worker kernel's chunk table: list of (tensor, first shard, start, length, padded offset,
    shard length when the chunk holds several shards else 0)."""
    count = ctypes.c_int64()
    _check(lib().onebit_adam_plan_worker_chunks(ctypes.byref(cfg), None, 0, ctypes.byref(count)),
           "onebit_adam_plan_worker_chunks")
    rows = (ctypes.c_int64 * (6 * max(count.value, 1)))()
    _check(lib().onebit_adam_plan_worker_chunks(ctypes.byref(cfg), rows, count.value, ctypes.byref(count)),
           "onebit_adam_plan_worker_chunks")
    return [tuple(rows[6 * q: 6 * q + 6]) for q in range(count.value)]


def _torch_dtype_code(dt) -> int:
    import torch

    return {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}[dt]


def _stream_ptr(stream=None) -> int:
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


class OneBitAdam:
    """1-bit Adam over a list of fp32 CUDA parameter tensors, with n simulated workers.

    Methods mirror the C ABI: ``warmup_step``, ``freeze_variance``, ``compress_step`` (gradients:
    list of n*T CUDA tensors ordered [worker][tensor]), their ``*_host`` variants (CPU tensors),
    ``get_status``, ``export_state``/``import_state``, ``comm_bytes``, timing helpers and ``free``.
    ``scale_block`` > 0 (a multiple of 32) gives every block of that many elements of a tensor its
    own worker scales and server shards (the per-chunk parameter-server form); scale exports are then
    indexed by block.
    """

    def __init__(self, params, n_workers, warmup_steps, beta1=0.9, beta2=0.999, eps=1e-8, lr=1e-3,
                 grad_dtype=None, bias_correction=False, workspace=None, stream=None, scale_block=0):
        import torch

        self.params = list(params)
        for p in self.params:
            if p.dtype != torch.float32 or not p.is_cuda or not p.is_contiguous():
                raise ValueError("parameters must be contiguous fp32 CUDA tensors")
        self.n = int(n_workers)
        self.T = len(self.params)
        self.numel = [p.numel() for p in self.params]
        gdt = F32 if grad_dtype is None else (grad_dtype if isinstance(grad_dtype, int) else _torch_dtype_code(grad_dtype))
        self.grad_dtype = gdt
        self.cfg = make_config(self.numel, self.n, warmup_steps, beta1, beta2, eps, lr, gdt, bias_correction,
                               scale_block)
        self.workspace = workspace
        ptrs = (ctypes.c_void_p * self.T)(*[p.data_ptr() for p in self.params])
        h = ctypes.c_void_p()
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        _check(lib().onebit_adam_init(ctypes.byref(self.cfg), ptrs, ws_ptr, ws_bytes, _stream_ptr(stream),
                                      ctypes.byref(h)), "onebit_adam_init")
        self.h = h

    # -------------------------------------------------------------- steps
    def _grad_array(self, grads, cuda=True, count=None):
        count = self.n * self.T if count is None else count  # [worker][tensor] pointers of `count` tensors
        if len(grads) != count:
            raise ValueError(f"expected {count} gradient tensors, got {len(grads)}")
        arr = (ctypes.c_void_p * len(grads))()
        for q, g in enumerate(grads):
            if g.is_cuda != cuda or not g.is_contiguous() or g.numel() != self.numel[q % self.T]:
                raise ValueError(f"gradient {q}: wrong device, layout or size")
            if _torch_dtype_code(g.dtype) != self.grad_dtype:
                raise ValueError(f"gradient {q}: dtype {g.dtype} does not match the config")
            arr[q] = g.data_ptr()
        return arr

    def warmup_step(self, grads, stream=None):
        _check(lib().onebit_adam_warmup_step(self.h, self._grad_array(grads), _stream_ptr(stream)),
               "onebit_adam_warmup_step", self.h)

    def freeze_variance(self, stream=None):
        _check(lib().onebit_adam_freeze_variance(self.h, _stream_ptr(stream)), "onebit_adam_freeze_variance", self.h)

    def compress_step(self, grads, stream=None):
        _check(lib().onebit_adam_compress_step(self.h, self._grad_array(grads), _stream_ptr(stream)),
               "onebit_adam_compress_step", self.h)

    def ec_adam_step(self, grads, stream=None):
        """Gradient-compression baseline step (1-bit EC compression of the gradients, then Adam)."""
        _check(lib().onebit_adam_ec_adam_step(self.h, self._grad_array(grads), _stream_ptr(stream)),
               "onebit_adam_ec_adam_step", self.h)

    def warmup_step_host(self, grads, stream=None):
        _check(lib().onebit_adam_warmup_step_host(self.h, self._grad_array(grads, cuda=False), _stream_ptr(stream)),
               "onebit_adam_warmup_step_host", self.h)

    def compress_step_host(self, grads, stream=None):
        _check(lib().onebit_adam_compress_step_host(self.h, self._grad_array(grads, cuda=False), _stream_ptr(stream)),
               "onebit_adam_compress_step_host", self.h)

    # -------------------------------------------------------------- status / state
    def get_status(self, stream=None) -> int:
        return int(lib().onebit_adam_get_status(self.h, _stream_ptr(stream)))

    def clear_status(self, stream=None):
        _check(lib().onebit_adam_clear_status(self.h, _stream_ptr(stream)), "onebit_adam_clear_status", self.h)

    def get_step(self):
        t, ph = ctypes.c_int64(), ctypes.c_int32()
        _check(lib().onebit_adam_get_step(self.h, ctypes.byref(t), ctypes.byref(ph)), "onebit_adam_get_step")
        return t.value, ph.value

    def set_step(self, t, phase, stream=None):
        _check(lib().onebit_adam_set_step(self.h, int(t), int(phase), _stream_ptr(stream)), "onebit_adam_set_step")

    def state_size(self, what) -> int:
        out = ctypes.c_size_t()
        _check(lib().onebit_adam_state_size(self.h, int(what), ctypes.byref(out)), "onebit_adam_state_size")
        return out.value

    def export_state(self, what, worker=0, stream=None):
        import torch

        nbytes = self.state_size(what)
        if what in (STATE_WORKER_BITS, STATE_SERVER_BITS):
            out = torch.empty(nbytes // 4, dtype=torch.int32, device=self.params[0].device)
        else:
            out = torch.empty(nbytes // 4, dtype=torch.float32, device=self.params[0].device)
        _check(lib().onebit_adam_export(self.h, int(what), int(worker), out.data_ptr(), _stream_ptr(stream)),
               "onebit_adam_export", self.h)
        return out

    def import_state(self, what, tensor, worker=0, stream=None):
        import torch

        # the copy is asynchronous on `stream`, so a temporary made here could be freed before it ran
        if (tensor.dtype != torch.float32 or not tensor.is_contiguous() or tensor.device != self.params[0].device
                or tensor.numel() * 4 != self.state_size(what)):
            raise ValueError("import expects a contiguous fp32 tensor of state_size bytes on the parameters' device")
        _check(lib().onebit_adam_import(self.h, int(what), int(worker), tensor.data_ptr(), _stream_ptr(stream)),
               "onebit_adam_import", self.h)

    def state_dict(self, stream=None):
        """Everything a resume needs besides the parameters (which the caller owns): the step count
        and phase, m, v (den after the freeze) and every error memory, in fp32 CUDA tensors."""
        t, phase = self.get_step()
        return {"t": t, "phase": phase,
                "m": self.export_state(STATE_M, stream=stream),
                "v": self.export_state(STATE_V, stream=stream),
                "server_error": self.export_state(STATE_SERVER_ERROR, stream=stream),
                "worker_error": [self.export_state(STATE_WORKER_ERROR, i, stream=stream) for i in range(self.n)]}

    def load_state_dict(self, d, stream=None):
        """Restore a state_dict() into this handle (same configuration): set_step, then the imports."""
        self.set_step(d["t"], d["phase"], stream=stream)
        self.import_state(STATE_M, d["m"], stream=stream)
        self.import_state(STATE_V, d["v"], stream=stream)
        self.import_state(STATE_SERVER_ERROR, d["server_error"], stream=stream)
        for i, e in enumerate(d["worker_error"]):
            self.import_state(STATE_WORKER_ERROR, e, i, stream=stream)

    def comm_bytes(self):
        c, f = ctypes.c_uint64(), ctypes.c_uint64()
        _check(lib().onebit_adam_comm_bytes(self.h, ctypes.byref(c), ctypes.byref(f)), "onebit_adam_comm_bytes")
        return c.value, f.value

    # -------------------------------------------------------------- timing
    def set_timing(self, enable: bool):
        _check(lib().onebit_adam_set_timing(self.h, int(bool(enable))), "onebit_adam_set_timing")

    def kernel_times(self):
        ms = (ctypes.c_double * NUM_KERNELS)()
        cnt = (ctypes.c_int64 * NUM_KERNELS)()
        _check(lib().onebit_adam_kernel_times(self.h, ms, cnt), "onebit_adam_kernel_times", self.h)
        return {KERNEL_NAMES[k]: (ms[k], cnt[k]) for k in range(NUM_KERNELS)}

    def set_lr(self, lr: float):
        """Learning rate for the following steps (for schedules; the method itself keeps it fixed)."""
        _check(lib().onebit_adam_set_lr(self.h, float(lr)), "onebit_adam_set_lr", self.h)

    def set_max_ctas(self, max_ctas: int):
        """Cap the CTAs of every streaming launch (0: fill the GPU); results do not depend on it."""
        _check(lib().onebit_adam_set_max_ctas(self.h, int(max_ctas)), "onebit_adam_set_max_ctas", self.h)

    def set_variance_monitor(self, enable: bool):
        _check(lib().onebit_adam_set_variance_monitor(self.h, int(bool(enable))), "onebit_adam_set_variance_monitor")

    def variance_norm(self):
        """(||v_t||_2, t) of the last monitored warm-up step (waits for it)."""
        v, t = ctypes.c_double(), ctypes.c_int64()
        _check(lib().onebit_adam_variance_norm(self.h, ctypes.byref(v), ctypes.byref(t)), "onebit_adam_variance_norm",
               self.h)
        return v.value, t.value

    def set_auto_freeze(self, tol: float):
        """The library's automatic freeze (0 turns it off): see onebit_adam_set_auto_freeze."""
        _check(lib().onebit_adam_set_auto_freeze(self.h, float(tol)), "onebit_adam_set_auto_freeze", self.h)

    def warmup_until_stable(self, grads_fn, tol: float, stream=None):
        """Warm-up steps with the library's automatic freeze on until the library freezes the
        variance (its norm's relative change per step at most `tol`, or T_w reached).  grads_fn(t)
        returns the gradients of warm-up step t (0-based).  Returns the steps taken."""
        t0, phase = self.get_step()
        t = t0
        self.set_auto_freeze(tol)
        try:
            while phase == PHASE_WARMUP:
                self.warmup_step(grads_fn(t), stream)
                t, phase = self.get_step()
        finally:
            self.set_auto_freeze(0.0)
        return t - t0

    def set_fault_injection(self, kind: int, value: int = 0):
        _check(lib().onebit_adam_set_fault_injection(self.h, int(kind), int(value)),
               "onebit_adam_set_fault_injection")

    def launch_count(self) -> int:
        out = ctypes.c_int64()
        _check(lib().onebit_adam_launch_count(self.h, ctypes.byref(out)), "onebit_adam_launch_count")
        return out.value

    def free(self):
        if getattr(self, "h", None):
            lib().onebit_adam_free(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.free()
        return False

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass
