"""onebit_worker_compress_noalloc: worker compression of one vector for callers that may not
allocate device memory (a framework's caching allocator owns every device byte, cudaMalloc's
implicit synchronisation is not acceptable in the caller's loop, or the caller is a plug-in with no
right to allocate).  Its scratch is a fixed device array inside the library, so the caller passes
only inputs and outputs.

Checked through the C ABI against the existing entry point, onebit_adam_compress_step, on a
one-worker handle: two calls in a row (the second fed the first's error output), each compared with
the handle's exported worker bits, scale and error after the matching compression step, with the
tolerances of the parity tests.  Checked against the oracle as well: c = (b1*m + (1-b1)*g) + err_in
formed in fp32 in that order, then the oracle's compressor ("1-bit Adam ...", Sec. 4.3: sign bits
and the magnitude-preserving scale, error = c - scale*sign(c)), over lengths from 1 to the maximum,
with the error updated in place, with unaligned pointers (the scalar path) and with no error input.
Collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import communication_compressed_optimizer_compress_gb300 as ob
import oracle
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


def _decode(g: torch.Tensor) -> np.ndarray:
    """Host fp32 values of a gradient tensor (every fp16 and bf16 value is exact in fp32)."""
    h = W.to_numpy_grad(g)
    if h.dtype == np.uint16:  # bfloat16 bits: the upper half of a binary32
        return (h.astype(np.uint32) << 16).view(np.float32)
    return h.astype(np.float32)


def _want(m, g, err_in, b1):
    """The oracle's worker compression of c = (b1*m + (1-b1)*g) + err_in, formed in fp32 in that order."""
    b1f = np.float32(b1)
    omb1 = np.float32(1.0) - b1f
    c = b1f * m + omb1 * g
    if err_in is not None:
        c = c + err_in
    s, words, err = oracle.compress(c)
    return c, s, words, err


def _view(buf: torch.Tensor, offset: int, n: int) -> torch.Tensor:
    return buf[offset: offset + n]


LENGTHS = [1, 7, 31, 33, 8 * 65536 + 5]
LAYOUTS = ["aligned", "in_place", "unaligned", "no_error_input"]


def _check_against_oracle(L, dtype, layout, seed):
    """Two calls in a row, the second continuing from the first one's error output; each compared
    with the oracle (sign bits exact outside the 1e-7*scale band, scale within 3e-7, error within
    1e-5 relative / 1e-7 absolute)."""
    dev = torch.device("cuda:0")
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    tdt = W.TORCH_DTYPE[dtype]
    off = 1 if layout == "unaligned" else 0  # one element into each allocation: the scalar path
    f = _entry()
    stream = torch.cuda.current_stream().cuda_stream
    b1 = 0.9
    m = _view(torch.randn(L + off, generator=gen, device=dev) * 1e-3, off, L)
    outs = [_view(torch.empty(L + off, device=dev), off, L) for _ in range(2)]
    err_in = None if layout == "no_error_input" else _view(torch.randn(L + off, generator=gen, device=dev) * 1e-4, off, L)
    nwords = (L + 31) // 32
    for call in range(2):
        err_out = err_in if layout == "in_place" else outs[call]
        g = _view((torch.randn(L + off, generator=gen, device=dev) * 1e-3).to(tdt), off, L)
        e_h = None if err_in is None else err_in.cpu().numpy().copy()
        c, s_want, w_want, err_want = _want(m.cpu().numpy(), _decode(g), e_h, b1)
        bits = torch.full((nwords,), -1, dtype=torch.int32, device=dev)  # garbage padding on purpose
        scale = torch.zeros(1, dtype=torch.float32, device=dev)
        rc = f(m.data_ptr(), g.data_ptr(), dtype, None if err_in is None else err_in.data_ptr(), b1, L,
               bits.data_ptr(), scale.data_ptr(), err_out.data_ptr(), stream)
        assert rc == ob.OK, ob.error_string(rc)
        torch.cuda.synchronize()
        got_s = float(scale.cpu()[0])
        assert abs(got_s - float(s_want)) <= 3e-7 * float(s_want), (L, call, got_s, s_want)
        keep = ~(np.abs(c.astype(np.float64)) < 1e-7 * float(s_want))
        got_w = bits.cpu().numpy()
        assert np.array_equal(_bits(got_w, L)[keep], _bits(w_want, L)[keep]), (L, call)
        if L % 32:
            assert int(got_w.view(np.uint32)[-1]) >> (L % 32) == 0, "padding bits must be 0"
        got_e = err_out.cpu().numpy().astype(np.float64)
        want_e = err_want.astype(np.float64)
        assert np.all(np.abs(got_e - want_e)[keep] <= 1e-7 + 1e-5 * np.abs(want_e[keep])), (L, call)
        err_in = err_out


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("L", LENGTHS)
@pytest.mark.parametrize("dtype", [W.F32, W.F16, W.BF16], ids=["f32", "f16", "bf16"])
def test_noalloc_matches_the_oracle(dtype, L, layout):
    _check_against_oracle(L, dtype, layout, seed=1000 + 7 * L + dtype + 31 * LAYOUTS.index(layout))


def test_noalloc_at_the_maximum_length():
    """The largest vector the fixed scratch array serves (2^28 elements: 4096 partials of 65536)."""
    _check_against_oracle(MAX_LEN, W.F16, "in_place", seed=77)


def test_noalloc_non_finite_input_reaches_the_scale():
    """A NaN gradient is not reported (the call returns before its kernels run): the scale is NaN."""
    dev = torch.device("cuda:0")
    L = 4096 + 3
    m = torch.zeros(L, device=dev)
    g = torch.full((L,), 1e-3, device=dev)
    g[100] = float("nan")
    bits = torch.zeros((L + 31) // 32, dtype=torch.int32, device=dev)
    scale = torch.zeros(1, device=dev)
    err = torch.empty(L, device=dev)
    rc = _entry()(m.data_ptr(), g.data_ptr(), W.F32, None, 0.9, L, bits.data_ptr(), scale.data_ptr(), err.data_ptr(),
                  torch.cuda.current_stream().cuda_stream)
    assert rc == ob.OK
    torch.cuda.synchronize()
    assert torch.isnan(scale).all()


def test_noalloc_rejects_overlapping_buffers():
    """Outputs that overlap an input or another output are refused before anything is enqueued."""
    f = _entry()
    dev = torch.device("cuda:0")
    L = 1000
    buf = torch.zeros(8 * L, device=dev)
    m, g, e_in, e_out = (buf[k * L:(k + 1) * L] for k in range(4))
    bits = torch.zeros(64, dtype=torch.int32, device=dev)
    scale = torch.zeros(2, device=dev)
    st = torch.cuda.current_stream().cuda_stream
    p = lambda t: t.data_ptr()  # noqa: E731
    ok = f(p(m), p(g), W.F32, p(e_in), 0.9, L, p(bits), p(scale), p(e_out), st)
    assert ok == ob.OK
    assert f(p(m), p(g), W.F32, p(e_out), 0.9, L, p(bits), p(scale), p(e_out), st) == ob.OK  # in place
    bad = [
        (p(m), p(g), p(e_in), p(bits), p(scale), p(m)),               # error output on the momentum
        (p(m), p(g), p(e_in), p(m), p(scale), p(e_out)),              # sign words on the momentum
        (p(m), p(g), p(e_in), p(bits), p(g) + 8, p(e_out)),           # scale inside the gradient
        (p(m), p(g), p(e_in), p(bits), p(e_out) + 40, p(e_out)),      # scale inside the error output
        (p(m), p(g), p(e_in), p(e_out) + 64, p(scale), p(e_out)),     # sign words inside the error output
        (p(m), p(g), p(e_in) + 4, p(bits), p(scale), p(e_in)),        # error in and out partly overlapping
        (p(m), p(g), p(e_in), p(bits), p(bits) + 16, p(e_out)),       # scale inside the sign words
    ]
    for args in bad:
        mm, gg, ee, bb, ss, oo = args
        assert f(mm, gg, W.F32, ee, 0.9, L, bb, ss, oo, st) == ob.ERR_INVALID_ARG, args
    torch.cuda.synchronize()
