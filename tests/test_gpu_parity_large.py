"""CUDA path vs the oracle at the chunk lengths the benchmark runs.

The launcher's chunk length grows with the element count (4096 for small lists, up to 65536 from
about 75e6 elements).  Short chunks never enter the worker kernel's batched main loop and give the
staged server kernel one tile per chunk, so these cases use lists large enough for chunks of 8192 to
65536 elements: multi-tile server chunks, the worker kernel's three-group loop, and (for the
full-size BERT-Base buffer and the 80e6-element BERT-Large-law buffer) exactly the kernels and chunk
length of the benchmark.  Every case is free-running (the oracle never sees a value computed by the
CUDA path) and compares every element after every step with the protocol of ``parity_util``, the
method's steps being those of "1-bit Adam: Communication Efficient Large-Scale Training with Adam's
Convergence Speed", Sec. 11 (worker error-compensated compression, server average and
recompression, broadcast and update).
"""
import pytest

import communication_compressed_optimizer_compress_gb300 as ob
from communication_compressed_optimizer_compress_gb300 import workloads as W
from parity_util import Pair

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SERVER_TILE = 4096  # elements per staged server tile


def _max_chunk(w):
    cfg = ob.make_config(list(w.numel), w.n_workers, w.warmup_steps, grad_dtype=w.grad_dtype)
    return max(r[3] for r in ob.plan_chunks(cfg)), max(r[3] for r in ob.plan_worker_chunks(cfg))


CASES = {
    # BERT-Large gradient law (log-uniform block sigma, fp16), 16 workers: chunks of 8192
    "f16_n16_d8M_block_sigma": W.WORKLOADS["bert_large"].with_(numel=(8_000_037,), warmup_steps=2,
                                                               compress_steps=3),
    # GPT-2 law (bf16, 1% of coordinates x100), 4 workers: chunks of 8192
    "bf16_n4_d6M_heavy_tail": W.WORKLOADS["gpt2_1p5b"].with_(numel=(6_000_011,), warmup_steps=2, compress_steps=3),
    # BERT-Base law (fp32 block sigma), 8 workers: chunks of 12288
    "f32_n8_d12M_block_sigma": W.WORKLOADS["bert_base"].with_(numel=(12_000_005,), warmup_steps=2,
                                                              compress_steps=3),
    # the first 16 tensors of the BERT-Large list (word and position embeddings, LayerNorm vectors,
    # the first layer), 8 workers, fp32: chunks of 40960, per-tensor scales
    "ragged_head_n8_f32": W.WORKLOADS["ragged_bert_large"].with_(numel=tuple(W.bert_large_shapes()[:16]),
                                                                 warmup_steps=2, compress_steps=3),
}


@pytest.mark.parametrize("name", list(CASES))
def test_large_chunks(name):
    w = CASES[name]
    cmax, wmax = _max_chunk(w)
    assert cmax > SERVER_TILE and wmax > SERVER_TILE, (cmax, wmax)
    p = Pair(w, gen_device="cuda")
    st = p.run()
    assert st.scales_exact >= 0.99 * st.scales, st
    limit = 1e-6 if w.law == "iid" else 1e-4  # small-sigma blocks sit closer to zero relative to the scale
    assert st.excluded_worker <= limit * st.worker_draws, st
    p.close()


FULL = {
    # the BERT-Base workload at its full size (110e6 fp32 parameters, 8 workers, fp32 block-sigma
    # gradients); two warm-up steps stand in for the hundred of the benchmark: the path is the same
    "bert_base_full": W.WORKLOADS["bert_base"].with_(warmup_steps=2, compress_steps=2),
    # the BERT-Large law (16 workers, fp16 block-sigma gradients) on 80e6 parameters: the benchmark's
    # kernels with its 65536-element chunks (16 server tiles per chunk)
    "bert_large_law_d80M": W.WORKLOADS["bert_large"].with_(numel=(80_000_000,), warmup_steps=1, compress_steps=2),
    # the GPT-2 law (4 workers, bf16 gradients with a 1% heavy tail) on 80e6 parameters: the 4-worker
    # kernel instances with 65536-element chunks
    "gpt2_law_d80M": W.WORKLOADS["gpt2_1p5b"].with_(numel=(80_000_000,), warmup_steps=1, compress_steps=2),
    # the 340-tensor BERT-Large list at full size (334e6 parameters, 8 workers, fp32, per-tensor scales)
    "ragged_bert_large_full": W.WORKLOADS["ragged_bert_large"].with_(warmup_steps=1, compress_steps=2),
    # the headline workload itself: BERT-Large, 340e6 parameters, 16 workers, fp16 block-sigma
    # gradients; one warm-up step stands in for the twenty of the benchmark (the path is the same),
    # then the first compression step and one steady-state step, every element compared
    "bert_large_full": W.WORKLOADS["bert_large"].with_(warmup_steps=1, compress_steps=2),
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_chunks(name):
    w = FULL[name]
    cmax, wmax = _max_chunk(w)
    assert cmax == 65536 and wmax == 65536, (cmax, wmax)
    p = Pair(w, gen_device="cuda")
    st = p.run()
    assert st.scales_exact >= 0.99 * st.scales, st
    assert st.excluded_worker <= 1e-4 * st.worker_draws, st
    p.close()


def test_baseline_step_at_the_benchmark_chunk_length():
    """The gradient-compression baseline ("1-bit Adam ...", Sec. 3.2 and 4.2: error-compensated 1-bit
    compression of the gradients, then Adam on the broadcast) on the BERT-Large law at 80e6 elements,
    16 workers, fp16: 65536-element chunks, two baseline steps (without and with error memories), a
    warm-up step, the freeze and a compression step, every element compared with the oracle."""
    w = W.WORKLOADS["bert_large"].with_(numel=(80_000_000,), warmup_steps=5)
    assert _max_chunk(w) == (65536, 65536)
    p = Pair(w, gen_device="cuda")
    for _ in range(2):
        p.ec_adam()
    p.warmup()
    p.freeze()
    p.compress()
    assert p.stats.scales_exact >= 0.99 * p.stats.scales, p.stats
    p.close()


def test_per_block_scales_at_size():
    """Per-block scales (the per-chunk parameter-server form of Sec. 11) with 65536-element blocks on
    the BERT-Large law at 24e6 elements, 16 workers: 4096-element shards, so the worker kernel's
    chunks each hold several whole shards (and look up each group's own broadcast scale); two
    compression steps compared element by element with the oracle."""
    w = W.WORKLOADS["bert_large"].with_(numel=(24_000_011,), warmup_steps=2, compress_steps=2)
    cfg = ob.make_config(list(w.numel), w.n_workers, w.warmup_steps, grad_dtype=w.grad_dtype, scale_block=65536)
    assert any(r[5] for r in ob.plan_worker_chunks(cfg))  # chunks spanning several shards
    p = Pair(w, scale_block=65536, gen_device="cuda")
    st = p.run()
    assert st.scales_exact >= 0.99 * st.scales, st
    p.close()


def test_short_scale_blocks_at_size():
    """Short scale blocks (4096 elements, n = 16: 256-element shards) on 2e6 elements of the BERT-Large
    law: worker chunks of one block each, holding sixteen shards, enough of them that the worker kernel
    runs one warp per unit; the update walks the same chunks and every scale is one partial.  Three
    compression steps compared element by element with the oracle ("1-bit Adam ...", Sec. 11)."""
    import torch

    w = W.WORKLOADS["bert_large"].with_(numel=(2_000_011,), warmup_steps=2, compress_steps=3)
    cfg = ob.make_config(list(w.numel), w.n_workers, w.warmup_steps, grad_dtype=w.grad_dtype, scale_block=4096)
    wrows = ob.plan_worker_chunks(cfg)
    assert any(r[5] for r in wrows) and max(r[3] for r in wrows) <= 8192  # spanning, short units
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert len(wrows) * w.n_workers >= 32 * sms  # enough units for one warp each
    p = Pair(w, scale_block=4096, gen_device="cuda")
    st = p.run()
    assert st.scales_exact >= 0.99 * st.scales, st
    p.close()
