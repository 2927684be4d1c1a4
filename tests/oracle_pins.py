"""Pins of the oracle to facts that do not come from the oracle itself.

Each ``pin_*`` function takes an ``oracle.OracleLib`` and raises AssertionError when the library
disagrees with a fact fixed by the pages or by mathematics: a worked example derived by hand from the
method's formulas (``tests/golden``), a closed form, an invariant the method states, a special case
that reduces to a textbook or library routine, or brute force on tiny inputs.  The same functions are
run against deliberately broken copies of the oracle (``test_oracle_mutants.py``) to show that a
plausible mistake anywhere in it fails at least one pin.

Sources: "1-bit Adam: Communication Efficient Large-Scale Training with Adam's Convergence Speed"
(Sec. 3.3, 4.1, 4.3, 6, 7.1, 11), the AIMech page "1-bit Adam (Two-Stage Preconditioner-Frozen
Error-Compensated Adam)" (summary formulas, gather-then-broadcast mechanism) and the codewithpapers
page "1-bit Adam" (scale definition, 97% / 94% volume reduction).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
F32, F16, BF16 = 0, 1, 2


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _ulp(x):
    return np.spacing(np.abs(np.float32(x))).astype(np.float64)


# ------------------------------------------------------------------------------ element helpers

def pin_half_decode(ora):
    """fp16 -> fp32 decoding equals numpy's IEEE binary16 conversion on all 65536 patterns."""
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([ora.half_to_float(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def pin_bf16_decode(ora):
    """bf16 -> fp32 decoding equals torch's bfloat16 conversion on all 65536 patterns."""
    import torch

    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = np.array([ora.bf16_to_float(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ------------------------------------------------------------------------------ the compressor

def pin_sign_word_layout(ora):
    """Hand-derived packed words (golden/sign_words.json): bit b of word w = element 32w+b."""
    gd = _golden("sign_words.json")
    v = np.ones(gd["length"], np.float32)
    v[gd["negatives"]] = -1.0
    v[gd["plus_zero"]] = 0.0
    v[gd["minus_zero"]] = -0.0
    want = np.array([int(h, 16) for h in gd["expected_words_hex"]], dtype=np.uint32)
    assert np.array_equal(ora.pack_signs(v), want)
    s, w, err = ora.compress(v.copy())
    assert np.array_equal(w, want)


def pin_pack_roundtrip_exhaustive(ora):
    """All 2^16 sign patterns of 16 elements survive pack -> unpack -> pack; NaN packs as 0."""
    for p in range(1 << 16):
        u = ora.unpack_signs(np.array([p], np.uint32), 16, 1.0)
        expect = np.where((p >> np.arange(16)) & 1, 1.0, -1.0).astype(np.float32)
        if not np.array_equal(u, expect):
            raise AssertionError(f"unpack pattern {p:#x}")
        if p % 257 == 0:  # re-pack a spread subset (pack is checked bit by bit below)
            assert int(ora.pack_signs(u)[0]) == p
    rng = np.random.default_rng(5)
    for length in range(1, 65):
        v = rng.standard_normal(length).astype(np.float32)
        w = ora.pack_signs(v)
        assert w.size == (length + 31) // 32
        bits = np.array([(int(w[e // 32]) >> (e % 32)) & 1 for e in range(length)])
        assert np.array_equal(bits, (v >= 0).astype(int))
        pad = length % 32
        if pad:
            assert int(w[-1]) >> pad == 0, "padding bits must be 0"
        back = ora.unpack_signs(w, length, 2.5)
        assert np.array_equal(back, np.where(v >= 0, 2.5, -2.5).astype(np.float32))
    assert int(ora.pack_signs(np.array([np.nan, -np.nan], np.float32))[0]) == 0


def pin_scale_preserves_magnitude(ora):
    """||scale * sign(c)||_2 = ||c||_2, i.e. sqrt(len) * scale = ||c||_2 (Sec. 4.3; codewithpapers)."""
    rng = np.random.default_rng(1)
    for length in (1, 2, 31, 33, 1000, 4097, 1 << 20):
        c = (rng.standard_normal(length) * rng.uniform(1e-6, 1e2)).astype(np.float32)
        s = float(ora.rms(c))
        ref = float(np.linalg.norm(c.astype(np.float64)))
        assert abs(math.sqrt(length) * s - ref) <= 2.0 ** -23 * ref, (length, s, ref)
        s2, w, err = ora.compress(c)
        assert float(s2) == s
    assert float(ora.rms(np.zeros(0, np.float32))) == 0.0
    assert float(ora.rms(np.zeros(7, np.float32))) == 0.0


def pin_scale_is_not_mean_abs(ora):
    """The magnitude-preserving scale differs from the L1 mean on a vector with unequal magnitudes."""
    c = np.array([3.0, -4.0, 0.0, 0.0], np.float32)   # ||c|| = 5, len 4 -> 2.5; mean |c| = 1.75
    assert float(ora.rms(c)) == 2.5


def pin_lossless_equal_magnitudes(ora):
    """Equal magnitudes compress losslessly: the error is exactly 0 when a is a power of two and
    within one ulp of a otherwise (Sec. 4.3: the 1-bit form keeps sign and magnitude)."""
    rng = np.random.default_rng(2)
    for length in (1, 5, 32, 33, 1000):
        for a in (0.25, 1.0, 2.0 ** -20, 3.0, 0.1, 7.3e-4):
            c = (np.where(rng.random(length) < 0.5, -1.0, 1.0) * a).astype(np.float32)
            s, w, err = ora.compress(c)
            if math.log2(a).is_integer():
                assert float(s) == float(np.float32(a)) and not np.any(err), (length, a)
            else:
                assert np.all(np.abs(err.astype(np.float64)) <= _ulp(a)), (length, a)


def pin_error_is_what_the_message_lost(ora):
    """The error memory is exactly c minus the decompressed message, zeros included (sign(0) = +1,
    so a zero element is sent as +scale and keeps -scale as its error)."""
    rng = np.random.default_rng(15)
    c = rng.standard_normal(300).astype(np.float32)
    c[[0, 7, 33, 64, 299]] = 0.0
    c[[5, 40]] = -0.0
    s, w, err = ora.compress(c)
    sent = ora.unpack_signs(w, c.size, float(s))
    assert np.array_equal(sent[[0, 5, 7, 33, 40, 64, 299]], np.full(7, s, np.float32))
    assert np.array_equal(err, c - sent)


def pin_error_statistics_gaussian(ora):
    """Gaussian c, large d: ||c - s sign(c)||^2 / ||c||^2 -> 2 - 2 sqrt(2/pi) (closed form for the
    magnitude-preserving scale; the L1-optimal scale would give 1 - 2/pi)."""
    rng = np.random.default_rng(3)
    d = 1 << 20
    c = rng.standard_normal(d).astype(np.float32)
    s, w, err = ora.compress(c)
    ratio = float(np.sum(err.astype(np.float64) ** 2) / np.sum(c.astype(np.float64) ** 2))
    assert abs(ratio - (2.0 - 2.0 * math.sqrt(2.0 / math.pi))) < 5.0 / math.sqrt(d), ratio


def pin_shard_rule(ora):
    """Server shards: n word-aligned pieces covering [0, L) in order, each at most S = 32 ceil(L/32n)."""
    for L in (0, 1, 5, 31, 32, 33, 64, 1000, 1 << 20, 110_000_000, 340_000_000, 1_560_000_000):
        for n in (1, 2, 3, 4, 8, 16):
            per = 32 * -(-L // (32 * n))
            prev = 0
            for j in range(n):
                lo, hi = ora.shard(L, n, j)
                assert lo == prev and lo <= hi <= L and hi - lo <= per and (lo % 32 == 0 or lo == L)
                prev = hi
            assert prev == L
    assert ora.shard(110_000_000, 8, 0) == (0, 13_750_016)
    assert ora.shard(110_000_000, 8, 7) == (7 * 13_750_016, 110_000_000)
    assert ora.shard(4, 2, 1) == (4, 4)


def pin_volume_reduction(ora):
    """Message size of a compressed vector (sign words + one fp32 scale) reproduces the pages'
    97% / 94% reduction and the 6% of the fp16 volume (golden/volume_reduction.json)."""
    gd = _golden("volume_reduction.json")["printed"]
    d = 340_000_000
    comp = 4 * ora.words(d) + 4
    r32 = 100.0 * (1.0 - comp / (4.0 * d))
    r16 = 100.0 * (1.0 - comp / (2.0 * d))
    frac16 = 100.0 * comp / (2.0 * d)
    assert abs(r32 - gd["reduction_vs_fp32_pct"]) <= 0.5
    assert abs(r16 - gd["reduction_vs_fp16_pct"]) <= 0.5
    assert abs(frac16 - gd["fraction_of_fp16_pct"]) <= 0.5


def pin_volume_reduction_including_warmup(ora):
    """The pages' 'up to 5x less communication, including the warm-up' from the message sizes: with
    the warm-up at f of the steps (uncompressed fp16 messages) and compressed messages after it, the
    run's volume falls by 1 / (f + (1 - f) * ratio).  Over the pages' 10-25% warm-up this spans the
    printed figure, and at 15% it is 5x (golden/volume_reduction.json)."""
    g = _golden("volume_reduction.json")
    d = 340_000_000
    ratio = (4 * ora.words(d) + 4) / (2.0 * d)
    total = lambda f: 1.0 / (f + (1.0 - f) * ratio)  # noqa: E731
    lo_f, hi_f = g["warmup_fraction_range"]
    printed = g["printed"]["total_reduction_including_warmup_x"]
    assert total(hi_f) < printed < total(lo_f)
    assert abs(total(0.15) - printed) <= 0.5


# ------------------------------------------------------------------------------ warm-up Adam

def pin_warmup_golden(ora):
    """Hand-worked warm-up step with eps = 0 (golden/warmup_step_eps0.json), with and without
    bias correction."""
    gd = _golden("warmup_step_eps0.json")
    c = gd["config"]
    for bc in (False, True):
        o = ora.optimizer(c["numel"], c["n_workers"], np.array(gd["x0"], np.float32), beta1=c["beta1"],
                          beta2=c["beta2"], eps=c["eps"], lr=c["lr"], bias_correction=bc)
        o.warmup_step([np.array(g, np.float32) for g in gd["grads"]])
        assert np.array_equal(o.view("m"), np.array(gd["expected"]["m"], np.float32))
        assert np.array_equal(o.view("v"), np.array(gd["expected"]["v"], np.float32))
        assert np.array_equal(o.view("x"), np.array(gd["expected"]["x"], np.float32))


def pin_warmup_constant_gradient_closed_form(ora):
    """Without bias correction and a constant gradient g: m_t = (1-b1^t) g, v_t = (1-b2^t) g^2 and
    x_T = x_0 - lr sum_t m_t / (sqrt(v_t) + eps)  (AIMech summary formulas, m_0 = v_0 = 0)."""
    rng = np.random.default_rng(4)
    d, n, T = 257, 3, 12
    b1, b2, eps, lr = 0.9, 0.999, 1e-8, 1e-3
    g = (rng.standard_normal(d) * 1e-3).astype(np.float32)
    x0 = (rng.standard_normal(d) * 0.02).astype(np.float32)
    o = ora.optimizer([d], n, x0, beta1=b1, beta2=b2, eps=eps, lr=lr)
    for _ in range(T):
        o.warmup_step([g] * n)
    B1, B2 = float(np.float32(b1)), float(np.float32(b2))
    gd = g.astype(np.float64)
    # the mean of n copies of g is g up to one rounding of the sum and one of the division
    mT = (1 - B1 ** T) * gd
    vT = (1 - B2 ** T) * gd * gd
    xT = x0.astype(np.float64).copy()
    for t in range(1, T + 1):
        xT -= float(np.float32(lr)) * ((1 - B1 ** t) * gd) / (np.sqrt((1 - B2 ** t) * gd * gd) + float(np.float32(eps)))
    assert np.allclose(o.view("m"), mT, rtol=1e-5, atol=0)
    assert np.allclose(o.view("v"), vT, rtol=1e-5, atol=0)
    assert np.allclose(o.view("x"), xT, rtol=1e-6, atol=1e-9)


def pin_warmup_matches_torch_adam(ora):
    """With bias correction, warm-up equals torch.optim.Adam (textbook Adam) on the mean gradient.
    Gradients are small dyadic numbers, so the mean of the n workers is exact on both sides; what
    is left is the two implementations' different rounding order."""
    import torch

    rng = np.random.default_rng(6)
    d, n, T = 1000, 4, 10
    x0 = (rng.standard_normal(d) * 0.02).astype(np.float32)
    o = ora.optimizer([d], n, x0, beta1=0.9, beta2=0.999, eps=1e-8, lr=1e-3, bias_correction=True)
    p = torch.nn.Parameter(torch.from_numpy(x0.copy()))
    # the hyper-parameters are fp32 numbers; torch gets the same values as doubles
    b1, b2 = float(np.float32(0.9)), float(np.float32(0.999))
    opt = torch.optim.Adam([p], lr=float(np.float32(1e-3)), betas=(b1, b2), eps=float(np.float32(1e-8)),
                           weight_decay=0.0)
    for _ in range(T):
        gs = [(rng.integers(-4096, 4096, d) / 2.0 ** 22).astype(np.float32) for _ in range(n)]
        o.warmup_step(gs)
        p.grad = torch.from_numpy((np.sum(np.stack(gs).astype(np.float64), axis=0) / n).astype(np.float32))
        opt.step()
    st = opt.state[p]
    m_ref, v_ref = st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()
    assert np.allclose(o.view("x"), p.detach().numpy(), rtol=1e-6, atol=1e-9)
    assert np.allclose(o.view("m"), m_ref, rtol=1e-6, atol=1e-6 * np.abs(m_ref).max())
    assert np.allclose(o.view("v"), v_ref, rtol=1e-6, atol=1e-6 * np.abs(v_ref).max())


def pin_warmup_mean_of_workers(ora):
    """Warm-up with n workers equals warm-up with one worker fed their exact mean (dyadic gradients,
    so the mean is exact): the allreduce of the uncompressed stage averages (Sec. 6)."""
    rng = np.random.default_rng(7)
    d, n = 64, 4
    gs = [(rng.integers(-64, 64, d) / 1024.0).astype(np.float32) for _ in range(n)]
    mean = (np.sum(np.stack(gs).astype(np.float64), axis=0) / n).astype(np.float32)
    x0 = np.zeros(d, np.float32)
    a = ora.optimizer([d], n, x0)
    b = ora.optimizer([d], 1, x0)
    for _ in range(3):
        a.warmup_step(gs)
        b.warmup_step([mean])
    for k in ("m", "v", "x"):
        assert np.array_equal(a.view(k), b.view(k)), k


def pin_variance_norm(ora):
    """||v||_2 of the warm-up variance: a 3-4-12-84 vector has norm 85 exactly; with a constant
    gradient g, ||v_t|| = (1 - b2^t) ||g^2|| (closed form of the summary formula for v_t)."""
    assert ora.norm2(np.array([3.0, 4.0, 12.0, 84.0], np.float32)) == 85.0
    assert ora.norm2(np.zeros(0, np.float32)) == 0.0
    rng = np.random.default_rng(16)
    d, T = 333, 9
    g = (rng.standard_normal(d) * 1e-2).astype(np.float32)
    o = ora.optimizer([d], 2, np.zeros(d, np.float32))
    B2 = float(np.float32(0.999))
    for t in range(1, T + 1):
        o.warmup_step([g, g])
        want = (1 - B2 ** t) * float(np.linalg.norm(g.astype(np.float64) ** 2))
        assert abs(ora.norm2(o.view("v")) - want) <= 1e-5 * want, t


def pin_freeze_closed_form(ora):
    """V = diag(sqrt(v_Tw) + eps); with bias correction v is divided by (1 - b2^Tw) first."""
    rng = np.random.default_rng(8)
    d = 500
    for bc in (False, True):
        o = ora.optimizer([d], 2, np.zeros(d, np.float32), bias_correction=bc, eps=1e-6)
        for _ in range(3):
            o.warmup_step([(rng.standard_normal(d) * 1e-2).astype(np.float32) for _ in range(2)])
        o.freeze()
        v = o.view("v").astype(np.float64)
        if bc:
            v = v / (1 - float(np.float32(0.999)) ** 3)
        want = np.sqrt(v) + float(np.float32(1e-6))
        assert np.allclose(o.view("den"), want, rtol=3e-7, atol=0)


# ------------------------------------------------------------------------------ compression stage

def _compress_ready(ora, numel, n, x0, den, m, **kw):
    o = ora.optimizer(numel, n, x0, **kw)
    o.t = 1
    o.phase = "compress"
    o.den[: o.D] = den
    o.m[: o.D] = m
    return o


def pin_compress_golden_n2(ora):
    """Hand-worked compression step, n = 2 (golden/compress_step_n2.json)."""
    gd = _golden("compress_step_n2.json")
    c = gd["config"]
    st = gd["state_before"]
    o = _compress_ready(ora, c["numel"], c["n_workers"], np.array(st["x"], np.float32),
                        np.array(st["den"], np.float32), np.array(st["m"], np.float32),
                        beta1=c["beta1"], beta2=c["beta2"], eps=c["eps"], lr=c["lr"])
    o.compress_step([np.array(g, np.float32) for g in gd["grads"]])
    ex = gd["expected"]
    assert np.array_equal(o.wscale, np.array(ex["wscale"], np.float32))
    assert np.array_equal(o.view("wbits"), np.array(ex["wbits"], np.uint32))
    assert np.array_equal(o.view("delta"), np.array(ex["delta"], np.float32))
    assert np.array_equal(o.sscale, np.array(ex["sscale"], np.float32))
    assert np.array_equal(o.view("sbits"), np.array(ex["sbits"], np.uint32))
    assert np.array_equal(o.view("eps_srv"), np.array(ex["eps_srv"], np.float32))
    assert np.array_equal(o.view("m"), np.array(ex["m"], np.float32))
    assert np.array_equal(o.view("x"), np.array(ex["x"], np.float32))


def _momentum_sgd_case(ora, n, identical):
    """Equal-magnitude momenta with a common sign pattern are compressed losslessly at the workers
    and at the server, so the compression stage reduces to momentum SGD with the coordinate-wise
    learning rate lr / (sqrt(v) + eps) (Sec. 3.3: once v is held fixed, each Adam step is a momentum
    step whose step size differs per coordinate)."""
    rng = np.random.default_rng(9 + n)
    d, steps = 96, 6
    sig = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    den = rng.uniform(0.5, 2.0, d).astype(np.float32)
    x0 = (rng.standard_normal(d) * 0.02).astype(np.float32)
    b1 = 0.5  # exact in fp32, so the closed form below is exact
    m = (sig * 0.25).astype(np.float32)
    o = _compress_ready(ora, [d], n, x0, den, m, beta1=b1, lr=2.0 ** -10)
    mref = m.astype(np.float64)
    xref = x0.astype(np.float64)
    for t in range(steps):
        if identical:
            mags = [2.0 ** -(t % 3)] * n
        else:
            mags = [2.0 ** -(t % 3) * (i + 1) for i in range(n)]
        gs = [(sig * mg).astype(np.float32) for mg in mags]
        o.compress_step(gs)
        gmean = sig * (sum(mags) / n)
        mref = b1 * mref + (1 - b1) * gmean
        xref = xref - (2.0 ** -10) * mref / den.astype(np.float64)
        assert np.allclose(o.view("m"), mref, rtol=1e-6, atol=0), t
        assert np.allclose(o.view("x"), xref, rtol=1e-6, atol=1e-9), t
        assert np.all(np.abs(o.view("delta")) <= 1e-6 * np.abs(mref).max()), t
        assert np.all(np.abs(o.view("eps_srv")) <= 1e-6 * np.abs(mref).max()), t


def pin_compress_reduces_to_momentum_sgd_n1(ora):
    _momentum_sgd_case(ora, 1, identical=True)


def pin_compress_reduces_to_momentum_sgd_identical_workers(ora):
    _momentum_sgd_case(ora, 4, identical=True)


def pin_compress_reduces_to_momentum_sgd_unequal_workers(ora):
    _momentum_sgd_case(ora, 3, identical=False)


def pin_server_scale_per_shard(ora):
    """n = 2, L = 64: shard 0 = [0, 32), shard 1 = [32, 64).  Worker signs agree on shard 0 and
    disagree on shard 1, so the server average is +-1 on shard 0 and 0 on shard 1: server scales 1
    and 0, and the broadcast momentum is +-1 then +0 (sign(0) = +1)."""
    d = 64
    rng = np.random.default_rng(11)
    sig = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    sig1 = sig.copy()
    sig1[32:] *= -1
    o = _compress_ready(ora, [d], 2, np.zeros(d, np.float32), np.ones(d, np.float32),
                        np.zeros(d, np.float32), beta1=0.5, lr=1.0)
    o.compress_step([(2 * sig).astype(np.float32), (2 * sig1).astype(np.float32)])
    assert np.array_equal(o.wscale, np.ones((2, 1), np.float32))
    assert np.array_equal(o.sscale, np.array([[1.0, 0.0]], np.float32))
    want_m = np.concatenate([sig[:32], np.zeros(32)]).astype(np.float32)
    assert np.array_equal(o.view("m"), want_m)
    assert np.array_equal(o.view("x"), -want_m)
    assert np.array_equal(np.signbit(o.view("m")[32:]), np.zeros(32, bool))


def _telescoping(ora, numel, n, steps, seed, dtype=F32):
    rng = np.random.default_rng(seed)
    D = sum(numel)
    x0 = (rng.standard_normal(D) * 0.02).astype(np.float32)
    den = rng.uniform(1e-3, 1e-1, D).astype(np.float32)
    m0 = (rng.standard_normal(D) * 1e-3).astype(np.float32)
    o = _compress_ready(ora, numel, n, x0, den, m0, grad_dtype=dtype)
    T = len(numel)
    sum_msg = np.zeros((n, D))
    sum_mi = np.zeros((n, D))
    sum_srv_out = np.zeros(D)
    sum_avg = np.zeros(D)
    b1, omb1 = np.float32(0.9), np.float32(1.0) - np.float32(0.9)
    offs = np.concatenate([[0], np.cumsum(numel)]).astype(int)
    woffs = np.concatenate([[0], np.cumsum([ora.words(L) for L in numel])]).astype(int)

    def unpack(words_row, scales_row):
        out = np.zeros(D)
        for k in range(T):
            L = numel[k]
            out[offs[k]: offs[k + 1]] = ora.unpack_signs(words_row[woffs[k]: woffs[k + 1]], L, scales_row[k])
        return out

    for t in range(steps):
        gs = []
        for i in range(n):
            flat = (rng.standard_normal(D) * 10 ** rng.uniform(-4, -2)).astype(np.float32)
            if dtype == F16:
                flat = flat.astype(np.float16)
            gs += [flat[offs[k]: offs[k + 1]] for k in range(T)]
        m_prev = o.view("m").copy()
        o.compress_step(gs)
        for i in range(n):
            g = np.concatenate(gs[i * T:(i + 1) * T]).astype(np.float32)
            mi = b1 * m_prev + omb1 * g          # the worker's local momentum of this step
            sum_mi[i] += mi
            msg = unpack(o.view("wbits")[i], o.wscale[i])
            sum_msg[i] += msg
        avg = np.zeros(D)
        for i in range(n):
            avg = avg + unpack(o.view("wbits")[i], o.wscale[i])
        avg = avg / n
        sum_avg += avg
        srv = np.zeros(D)
        for k in range(T):
            L = numel[k]
            for j in range(n):
                lo, hi = ora.shard(L, n, j)
                w = o.view("sbits")[woffs[k]: woffs[k + 1]]
                full = ora.unpack_signs(w, L, o.sscale[k, j])
                srv[offs[k] + lo: offs[k] + hi] = full[lo:hi]
        sum_srv_out += srv
        # the broadcast result is the shared momentum
        assert np.array_equal(o.view("m").astype(np.float64), srv)
    # error feedback telescopes (Sec. 4.1): sum of messages + final error = sum of inputs
    for i in range(n):
        lhs = sum_msg[i] + o.view("delta")[i]
        scale = np.abs(sum_mi[i]).max() + 1e-30
        assert np.max(np.abs(lhs - sum_mi[i])) <= 1e-6 * scale * steps, i
    lhs = sum_srv_out + o.view("eps_srv")
    scale = np.abs(sum_avg).max() + 1e-30
    assert np.max(np.abs(lhs - sum_avg)) <= 1e-6 * scale * steps


def pin_error_feedback_telescopes_flat(ora):
    """Worker and server error feedback telescope over steps: sum of messages + final error = sum of
    the compressed inputs, to 1e-6 relative (Sec. 4.1 / AIMech delta and epsilon memories)."""
    _telescoping(ora, [1000], 3, 6, 12)


def pin_error_feedback_telescopes_ragged_f16(ora):
    _telescoping(ora, [5, 0, 33, 200], 4, 5, 13, dtype=F16)


def pin_tensors_are_independent(ora):
    """Per-tensor scales and shards make the tensors of a list independent problems: stepping the
    list equals stepping each tensor alone (brute force on small ragged sizes)."""
    rng = np.random.default_rng(14)
    numel = [1, 5, 32, 33, 0, 70]
    n = 3
    D = sum(numel)
    x0 = (rng.standard_normal(D) * 0.02).astype(np.float32)
    whole = ora.optimizer(numel, n, x0)
    parts = []
    off = 0
    for L in numel:
        parts.append(ora.optimizer([L], n, x0[off: off + L]))
        off += L
    for step in range(7):
        gs_flat = [(rng.standard_normal(D) * 1e-3).astype(np.float32) for _ in range(n)]
        offs = np.concatenate([[0], np.cumsum(numel)]).astype(int)
        gs = [gs_flat[i][offs[k]: offs[k + 1]] for i in range(n) for k in range(len(numel))]
        if step < 3:
            whole.warmup_step(gs)
        else:
            whole.compress_step(gs)
        for k, p in enumerate(parts):
            gk = [gs_flat[i][offs[k]: offs[k + 1]] for i in range(n)]
            if step < 3:
                p.warmup_step(gk)
            else:
                p.compress_step(gk)
        if step == 2:
            whole.freeze()
            for p in parts:
                p.freeze()
    xs = np.concatenate([p.view("x") for p in parts])
    assert np.array_equal(whole.view("x"), xs)
    for k, p in enumerate(parts):
        assert np.array_equal(whole.wscale[:, k], p.wscale[:, 0])
        assert np.array_equal(whole.sscale[k], p.sscale[0])


def pin_scale_blocks_lossless_on_blockwise_magnitudes(ora):
    """Per-chunk scale granularity ("1-bit Adam ...", Sec. 11: compression per chunk).  When every
    block of B elements holds one magnitude (random signs), a per-block scale sends it exactly: the
    worker and server errors stay 0, every scale equals that block's |c|, and the update is the
    uncompressed momentum step.  The same input with one scale per tensor is lossy."""
    import oracle as _o
    numel, B, n = [224, 0, 96], 64, 2
    assert _o.scale_blocks(numel, B) == [64, 64, 64, 32, 0, 64, 32]
    assert _o.scale_blocks(numel, 0) == numel
    rng = np.random.default_rng(21)
    D = sum(numel)
    x0 = (rng.standard_normal(D) * 0.1).astype(np.float32)
    b1, lr = np.float32(0.75), np.float32(0.5)
    mags = np.float32(2.0) ** np.arange(-6, 1).astype(np.float32)  # one per block
    blk_of = np.concatenate([np.full(L, b) for b, L in enumerate(_o.scale_blocks(numel, B))]).astype(int)
    g = (mags[blk_of] * np.where(rng.random(D) < 0.5, -1, 1)).astype(np.float32)
    offs = np.concatenate([[0], np.cumsum(numel)]).astype(int)
    per_tensor = [g[offs[k]: offs[k + 1]] for k in range(len(numel))]
    zeros = [np.zeros(L, np.float32) for L in numel]
    results = {}
    for blk in (B, 0):
        o = ora.optimizer(numel, n, x0, beta1=b1, eps=1.0, lr=lr, scale_block=blk)
        o.warmup_step(zeros * n)         # m = v = 0, so den = 0 + eps = 1 after the freeze
        o.freeze()
        o.compress_step(per_tensor * n)  # identical workers
        results[blk] = o
    o = results[B]
    c = (np.float32(1) - b1) * g
    assert np.all(o.view("delta") == 0) and np.all(o.view("eps_srv") == 0)
    for b, L in enumerate(_o.scale_blocks(numel, B)):
        want = np.float32((np.float32(1) - b1) * mags[b]) if L else np.float32(0)
        assert o.wscale[0, b] == want and o.wscale[1, b] == want
        for j in range(n):
            lo, hi = ora.shard(L, n, j)
            assert o.sscale[b, j] == (want if hi > lo else 0)
    assert np.array_equal(o.view("m"), c)
    assert np.array_equal(o.view("x"), x0 - lr * c)
    assert np.abs(results[0].view("delta")).max() > 0.1 * np.abs(c).max()


def pin_scale_block_larger_than_tensors_is_per_tensor(ora):
    """A block at least as long as every tensor leaves each tensor one block: the per-tensor method."""
    rng = np.random.default_rng(22)
    numel, n = [40, 0, 200, 7], 3
    D = sum(numel)
    x0 = (rng.standard_normal(D) * 0.05).astype(np.float32)
    a = ora.optimizer(numel, n, x0)
    b = ora.optimizer(numel, n, x0, scale_block=256)
    assert b.numel == numel
    offs = np.concatenate([[0], np.cumsum(numel)]).astype(int)
    for step in range(6):
        gf = [(rng.standard_normal(D) * 1e-2).astype(np.float32) for _ in range(n)]
        gs = [gf[i][offs[k]: offs[k + 1]] for i in range(n) for k in range(len(numel))]
        for o in (a, b):
            if step < 2:
                o.warmup_step(gs)
            else:
                o.compress_step(gs)
            if step == 1:
                o.freeze()
    for name in ("x", "m", "delta", "eps_srv", "wbits", "sbits", "wscale", "sscale"):
        assert np.array_equal(a.view(name), b.view(name)), name


def pin_scale_blocks_equal_presplit_tensors(ora):
    """Cutting tensors into blocks inside the optimizer equals handing it the blocks as separate
    tensors (random data, ragged blocks, several workers and steps): the blocking is only a view."""
    rng = np.random.default_rng(23)
    numel, B, n = [300, 5, 0, 129], 64, 3
    import oracle as _o
    blocks = _o.scale_blocks(numel, B)
    D = sum(numel)
    x0 = (rng.standard_normal(D) * 0.05).astype(np.float32)
    a = ora.optimizer(numel, n, x0, scale_block=B)
    b = ora.optimizer(blocks, n, x0)
    offs = np.concatenate([[0], np.cumsum(numel)]).astype(int)
    boffs = np.concatenate([[0], np.cumsum(blocks)]).astype(int)
    for step in range(6):
        gf = [(rng.standard_normal(D) * 1e-2).astype(np.float32) for _ in range(n)]
        ga = [gf[i][offs[k]: offs[k + 1]] for i in range(n) for k in range(len(numel))]
        gb = [gf[i][boffs[k]: boffs[k + 1]] for i in range(n) for k in range(len(blocks))]
        for o, gs in ((a, ga), (b, gb)):
            if step < 2:
                o.warmup_step(gs)
            else:
                o.compress_step(gs)
            if step == 1:
                o.freeze()
    for name in ("x", "m", "delta", "eps_srv", "wbits", "sbits", "wscale", "sscale"):
        assert np.array_equal(a.view(name), b.view(name)), name


def pin_ec_adam_lossless_is_adam(ora):
    """Baseline of Sec. 3.2 (1-bit EC compression of the gradients, then Adam): when every worker's
    gradient has equal magnitudes and all share one sign pattern, worker and server compression are
    lossless, so the step is textbook Adam (torch.optim.Adam, bias-corrected) on the mean gradient."""
    import torch

    rng = np.random.default_rng(17)
    d, n, T = 256, 4, 6
    sig = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    x0 = (rng.standard_normal(d) * 0.02).astype(np.float32)
    o = ora.optimizer([d], n, x0, beta1=0.9, beta2=0.999, eps=1e-8, lr=1e-3, bias_correction=True)
    p = torch.nn.Parameter(torch.from_numpy(x0.copy()))
    b1, b2 = float(np.float32(0.9)), float(np.float32(0.999))
    opt = torch.optim.Adam([p], lr=float(np.float32(1e-3)), betas=(b1, b2), eps=float(np.float32(1e-8)))
    for t in range(T):
        mags = [2.0 ** -(8 + (t + i) % 3) for i in range(n)]
        gs = [(sig * a).astype(np.float32) for a in mags]
        o.ec_adam_step(gs)
        p.grad = torch.from_numpy((sig * (sum(mags) / n)).astype(np.float32))
        opt.step()
        assert not np.any(o.view("delta")) and not np.any(o.view("eps_srv")), t
    assert np.allclose(o.view("x"), p.detach().numpy(), rtol=1e-6, atol=1e-9)
    assert np.allclose(o.view("m"), opt.state[p]["exp_avg"].numpy(), rtol=1e-6, atol=0)
    assert np.allclose(o.view("v"), opt.state[p]["exp_avg_sq"].numpy(), rtol=1e-6, atol=0)


def pin_ec_adam_error_feedback_telescopes(ora):
    """The baseline's error feedback telescopes on the gradients: sum of messages + final error =
    sum of gradients (workers), and likewise for the server (Sec. 4.1)."""
    rng = np.random.default_rng(18)
    numel = [300, 0, 65]
    D, n, T, steps = sum(numel), 3, len(numel), 5
    offs = np.concatenate([[0], np.cumsum(numel)]).astype(int)
    woffs = np.concatenate([[0], np.cumsum([ora.words(L) for L in numel])]).astype(int)
    o = ora.optimizer(numel, n, np.zeros(D, np.float32))

    def decode(words_row, scales_row):
        out = np.zeros(D)
        for k, L in enumerate(numel):
            out[offs[k]: offs[k + 1]] = ora.unpack_signs(words_row[woffs[k]: woffs[k + 1]], L, scales_row[k])
        return out

    sum_g = np.zeros((n, D))
    sum_msg = np.zeros((n, D))
    sum_avg = np.zeros(D)
    sum_srv = np.zeros(D)
    for _ in range(steps):
        flats = [(rng.standard_normal(D) * 1e-3).astype(np.float32) for _ in range(n)]
        o.ec_adam_step([f[offs[k]: offs[k + 1]] for f in flats for k in range(T)])
        avg = np.zeros(D)
        for i in range(n):
            sum_g[i] += flats[i]
            msg = decode(o.view("wbits")[i], o.wscale[i])
            sum_msg[i] += msg
            avg += msg
        avg /= n
        sum_avg += avg
        srv = np.zeros(D)
        for k, L in enumerate(numel):
            w = o.view("sbits")[woffs[k]: woffs[k + 1]]
            for j in range(n):
                lo, hi = ora.shard(L, n, j)
                srv[offs[k] + lo: offs[k] + hi] = ora.unpack_signs(w, L, o.sscale[k, j])[lo:hi]
        sum_srv += srv
    for i in range(n):
        scale = np.abs(sum_g[i]).max()
        assert np.max(np.abs(sum_msg[i] + o.view("delta")[i] - sum_g[i])) <= 1e-6 * scale * steps, i
    assert np.max(np.abs(sum_srv + o.view("eps_srv") - sum_avg)) <= 1e-6 * np.abs(sum_avg).max() * steps


def _brute_rms(vals):
    """||v||_2 / sqrt(len) from the correctly rounded sum of the exact squares (math.fsum), taken in
    double and rounded once to fp32; 0 for an empty range."""
    if not vals:
        return np.float32(0.0)
    return np.float32(math.sqrt(math.fsum(float(v) * float(v) for v in vals) / len(vals)))


def pin_brute_force_whole_algorithm_small_d(ora):
    """The whole method on tiny inputs, restated here element by element in scalar fp32 from its
    steps.  Warm-up Adam runs on the ordered mean of the worker gradients, with or without
    Kingma-Ba correction.  The freeze gives den = sqrt(v) + eps.  Each compression step then runs
    worker momentum, error compensation, sign + rms scale per tensor, the ordered server average,
    the server error, per-shard recompression, the broadcast and the preconditioned update.
    Shards are 32*ceil(L/(32n)) and norms come from exactly rounded sums.  Every state word must
    equal the oracle's after every step.  Cases: the ragged list {1, 5, 32, 33} at
    n in {1, 2, 3, 4, 8}, an empty tensor, a single 64-element tensor, zero gradients
    (sign(0) = +1), and fp32, fp16 and bf16 gradients."""
    cases = [([64], 1, F32, False), ([1, 5, 32, 33], 2, F32, False), ([1, 5, 32, 33], 3, F16, True),
             ([1, 5, 32, 33], 4, BF16, False), ([1, 5, 32, 33], 8, F32, False), ([33, 0, 31], 5, F32, True),
             ([64], 3, F32, False)]
    T_w, steps = 2, 4
    for case, (numel, n, dtype, bc) in enumerate(cases):
        rng = np.random.default_rng(300 + case)
        D, T = sum(numel), len(numel)
        offs = np.concatenate([[0], np.cumsum(numel)]).astype(int)
        b1, b2, eps_adam, lr = np.float32(0.9), np.float32(0.999), np.float32(1e-8), np.float32(1e-2)
        one = np.float32(1.0)
        omb1, omb2 = np.float32(one - b1), np.float32(one - b2)
        x0 = (rng.standard_normal(D) * 0.02).astype(np.float32)
        x = list(x0)
        m = [np.float32(0.0)] * D
        v = [np.float32(0.0)] * D
        o = ora.optimizer(numel, n, x0, beta1=float(b1), beta2=float(b2), eps=float(eps_adam), lr=float(lr),
                          grad_dtype=dtype, bias_correction=bc)

        def draw(zero_head):
            flats, vals = [], []
            for _ in range(n):
                f = (rng.standard_normal(D) * 10 ** rng.uniform(-4, -2)).astype(np.float32)
                if zero_head:
                    f[: D // 4] = 0.0
                if dtype == F16:
                    f = f.astype(np.float16)
                    vals.append([np.float32(e) for e in f])
                elif dtype == BF16:
                    f = (f.view(np.uint32) >> 16).astype(np.uint16)  # truncated to bf16 bits
                    vals.append([(np.uint32(e) << np.uint32(16)).view(np.float32) for e in f])
                else:
                    vals.append(list(f))
                flats.append(f)
            return [f[offs[k]: offs[k + 1]] for f in flats for k in range(T)], vals

        def check(name, want, where):
            got = o.view(name)
            assert np.array_equal(got.view(np.uint32), np.array(want, np.float32).view(np.uint32)), (where, name)

        # warm-up: Adam on the ordered mean of the n gradients
        for t in range(1, T_w + 1):
            grads, g = draw(False)
            o.warmup_step(grads)
            bc1 = np.float32(1.0 - float(b1) ** t)
            bc2 = np.float32(1.0 - float(b2) ** t)
            for p in range(D):
                acc = np.float32(0.0)
                for i in range(n):
                    acc = np.float32(acc + g[i][p])
                gm = np.float32(acc / np.float32(n))
                m[p] = np.float32(np.float32(b1 * m[p]) + np.float32(omb1 * gm))
                v[p] = np.float32(np.float32(b2 * v[p]) + np.float32(omb2 * np.float32(gm * gm)))
                mh, vh = (np.float32(m[p] / bc1), np.float32(v[p] / bc2)) if bc else (m[p], v[p])
                x[p] = np.float32(x[p] - np.float32(lr * np.float32(mh / np.float32(np.sqrt(vh) + eps_adam))))
            for name, want in (("x", x), ("m", m), ("v", v)):
                check(name, want, f"case {case} warm-up {t}")

        # freeze: den = sqrt(v) + eps (v bias-corrected at t = T_w when correction is on)
        o.freeze()
        bc2 = np.float32(1.0 - float(b2) ** T_w)
        den = [np.float32(np.sqrt(np.float32(v[p] / bc2) if bc else v[p]) + eps_adam) for p in range(D)]
        check("den", den, f"case {case} freeze")
        delta = [[np.float32(0.0)] * D for _ in range(n)]
        eps = [np.float32(0.0)] * D

        for step in range(steps):
            grads, g = draw(step == 0)
            o.compress_step(grads)

            # worker i: m_i = b1*m + (1-b1)*g_i, c_i = m_i + delta_i, then sign + scale per tensor
            wscale = np.zeros((n, T), np.float32)
            msg = [[None] * D for _ in range(n)]
            wbits = [[0] * D for _ in range(n)]
            for i in range(n):
                c = [np.float32(np.float32(b1 * m[p]) + np.float32(omb1 * g[i][p])) for p in range(D)]
                c = [np.float32(c[p] + delta[i][p]) for p in range(D)]
                for k in range(T):
                    sc = _brute_rms(c[offs[k]: offs[k + 1]])
                    wscale[i, k] = sc
                    for p in range(offs[k], offs[k + 1]):
                        bit = c[p] >= 0
                        wbits[i][p] = int(bit)
                        msg[i][p] = sc if bit else -sc
                        delta[i][p] = np.float32(c[p] - sc) if bit else np.float32(c[p] + sc)
            # server: ordered sum of the messages, / n, + server error; recompress per shard
            a = []
            for p in range(D):
                acc = np.float32(0.0)
                for i in range(n):
                    acc = np.float32(acc + msg[i][p])
                a.append(np.float32(np.float32(acc / np.float32(n)) + eps[p]))
            sscale = np.zeros((T, n), np.float32)
            sbits = [0] * D
            for k, L in enumerate(numel):
                S_k = 32 * -(-L // (32 * n))
                for j in range(n):
                    lo, hi = offs[k] + min(j * S_k, L), offs[k] + min((j + 1) * S_k, L)
                    S = _brute_rms(a[lo:hi])
                    sscale[k, j] = S
                    for p in range(lo, hi):
                        bit = a[p] >= 0
                        sbits[p] = int(bit)
                        eps[p] = np.float32(a[p] - S) if bit else np.float32(a[p] + S)
                        m[p] = S if bit else -S
            x = [np.float32(x[p] - np.float32(lr * np.float32(m[p] / den[p]))) for p in range(D)]

            def words(bits):
                out = []
                for k, L in enumerate(numel):
                    for w0 in range(0, L, 32):
                        out.append(sum(bits[offs[k] + e] << (e - w0) for e in range(w0, min(w0 + 32, L))))
                return np.array(out, np.uint32)

            where = f"case {case} compression step {step}"
            assert np.array_equal(o.wscale, wscale), where
            assert np.array_equal(o.sscale, sscale), where
            for i in range(n):
                assert np.array_equal(o.view("wbits")[i], words(wbits[i])), where
                got = o.view("delta")[i].view(np.uint32)
                assert np.array_equal(got, np.array(delta[i], np.float32).view(np.uint32)), where
            assert np.array_equal(o.view("sbits"), words(sbits)), where
            for name, want in (("eps_srv", eps), ("m", m), ("x", x)):
                check(name, want, where)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
