"""onebit_worker_compress_noalloc: worker compression of one vector for callers that may not
allocate device memory (a framework's caching allocator owns every device byte, cudaMalloc's
implicit synchronisation is not acceptable in the caller's loop, or the caller is a plug-in with no
right to allocate).  Its scratch is a fixed device array inside the library, so the caller passes
only inputs and outputs.

Checked through the C ABI against the existing entry point, onebit_adam_compress_step, on a
one-worker handle: two calls in a row (the second fed the first's error output), each compared with
the handle's exported worker bits, scale and error after the matching compression step, with the
tolerances of the parity tests.  Collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import communication_compressed_optimizer_compress_gb300 as ob
from communication_compressed_optimizer_compress_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_LEN = 268435456  # ONEBIT_NOALLOC_MAX_LEN in include/onebit_adam.h


def _entry():
    f = ob.lib().onebit_worker_compress_noalloc
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, ctypes.c_int32, vp, ctypes.c_float, ctypes.c_int64, vp, vp, vp, vp]
    f.restype = ctypes.c_int
    return f


def _bits(words, length):
    w = words.view(np.uint32)
    return ((w[:, None] >> np.arange(32, dtype=np.uint32)[None, :]) & 1).astype(bool).reshape(-1)[:length]


@pytest.mark.parametrize("dtype", [W.F32, W.F16, W.BF16], ids=["f32", "f16", "bf16"])
def test_noalloc_matches_compress_step(dtype):
    L = 3 * 65536 + 1237  # several chunks and a ragged last word
    w = W.WORKLOADS["tiny"].with_(numel=(L,), n_workers=1, grad_dtype=dtype, warmup_steps=2, seed=91)
    dev = torch.device("cuda:0")
    params = [p.to(dev) for p in W.params(w, "cpu")]
    opt = ob.OneBitAdam(params, 1, w.warmup_steps, w.beta1, w.beta2, w.eps, w.lr, grad_dtype=W.TORCH_DTYPE[dtype])
    src = W.GradSource(w, "cpu")
    for s in range(w.warmup_steps):
        opt.warmup_step([g.to(dev) for g in src.grads(s)])
    opt.freeze_variance()
    f = _entry()
    stream = torch.cuda.current_stream().cuda_stream
    err_in = None
    nwords = (L + 31) // 32
    for call in range(2):
        m_before = opt.export_state(ob.STATE_M)  # the shared momentum the step starts from
        g = src.grads(w.warmup_steps + call)[0].to(dev)
        opt.compress_step([g])
        want_bits = opt.export_state(ob.STATE_WORKER_BITS, 0).cpu().numpy()
        want_scale = float(opt.export_state(ob.STATE_WORKER_SCALES).cpu()[0])
        want_err = opt.export_state(ob.STATE_WORKER_ERROR, 0).cpu().numpy()

        bits = torch.full((nwords,), -1, dtype=torch.int32, device=dev)  # garbage padding on purpose
        scale = torch.zeros(1, dtype=torch.float32, device=dev)
        err_out = torch.empty(L, dtype=torch.float32, device=dev)
        rc = f(m_before.data_ptr(), g.data_ptr(), dtype, None if err_in is None else err_in.data_ptr(),
               w.beta1, L, bits.data_ptr(), scale.data_ptr(), err_out.data_ptr(), stream)
        assert rc == ob.OK, ob.error_string(rc)
        torch.cuda.synchronize()
        got_bits = bits.cpu().numpy()
        got_scale = float(scale.cpu()[0])
        got_err = err_out.cpu().numpy()

        assert abs(got_scale - want_scale) <= 3e-7 * want_scale, (got_scale, want_scale)
        wb = _bits(want_bits, L)
        c_want = want_err.astype(np.float64) + np.where(wb, want_scale, -want_scale)
        keep = ~(np.abs(c_want) < 1e-7 * want_scale)
        assert np.array_equal(_bits(got_bits, L)[keep], wb[keep])
        assert int(got_bits.view(np.uint32)[-1]) >> (L % 32) == 0, "padding bits must be 0"
        diff = np.abs(got_err.astype(np.float64) - want_err)[keep]
        assert np.all(diff <= 1e-7 + 1e-5 * np.abs(want_err[keep].astype(np.float64)))
        err_in = err_out  # the second call continues from the first call's error
    opt.free()


def test_noalloc_rejects_sizes_beyond_the_limit():
    f = _entry()
    buf = torch.zeros(64, dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    stream = torch.cuda.current_stream().cuda_stream
    assert f(p, p, W.F32, None, 0.9, MAX_LEN + 1, p, p, p, stream) == ob.ERR_INVALID_ARG
    assert f(p, p, W.F32, None, 0.9, 0, p, p, p, stream) == ob.ERR_INVALID_ARG
    assert f(None, p, W.F32, None, 0.9, 16, p, p, p, stream) == ob.ERR_INVALID_ARG
