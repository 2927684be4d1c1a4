"""Seeded synthetic inputs for the 1-bit Adam optimizer step.

This module holds only input recipes (sizes, value distributions, seeds).  It contains none of the
method's arithmetic, so both the CUDA path's callers and the oracle's callers can draw from it.

The pages train BERT-Base, BERT-Large and GPT-2 on real corpora ("1-bit Adam ...", Sec. 7 and
Sec. 7.1); no dataset or trained weight is used here.  Synthetic parameter and gradient buffers of
those models' sizes stand in for them:

* ``tiny``: one flat fp32 buffer of 2^20 parameters, n=4 workers; params ~ N(0, 0.02^2),
  per-worker gradients iid N(0, (1e-3)^2), fresh every step; 5 warm-up Adam steps, 5 compression steps.
* ``bert_base``: flat buffer of 110e6 fp32 parameters, n=8; gradients fp32 sigma_k * N(0,1) where
  sigma_k = 10^U(-5,-2) is drawn once per block of 2^20 elements and shared by all workers and steps.
* ``bert_large``: flat buffer of 340e6, n=16, same gradient law rounded to fp16 (subnormals kept).
* ``ragged_bert_large``: the 340-tensor BERT-Large parameter list (word embedding 30522x1024,
  position 512x1024, embedding LayerNorm 2x1024, 24 layers of QKV 1024x3072, output 1024x1024,
  FFN 1024x4096 and 4096x1024 plus their bias and LayerNorm vectors), n=8, fp32 gradients N(0,(1e-3)^2).
* ``gpt2_1p5b``: flat buffer of 1.56e9, n=4, bf16 gradients N(0,(1e-3)^2) with a fixed 1% of the
  coordinates (drawn once) multiplied by 100 (heavy tail).

"N(0, s)" in the workload text is read with s as the standard deviation.

One more law serves the parity tests of the norms' range: ``tensor_std`` gives tensor k gradients
N(0, tensor_std[k]^2), so that whole tensors sit at extreme magnitudes (1e-30, 1e25, ...).
"""
from __future__ import annotations

import dataclasses
import math

import torch

F32, F16, BF16 = 0, 1, 2
TORCH_DTYPE = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}
GRAD_BYTES = {F32: 4, F16: 2, BF16: 2}
DTYPE_NAME = {F32: "f32", F16: "f16", BF16: "bf16"}


def bert_large_shapes() -> list[int]:
    """numel of every tensor of the BERT-Large parameter list (340 tensors)."""
    h, ff, layers = 1024, 4096, 24
    out = [30522 * h, 512 * h, h, h]            # word, position embeddings; embedding LayerNorm
    for _ in range(layers):
        out += [h * 3 * h, h, h, h]             # QKV weight; Q, K, V biases
        out += [h * h, h]                       # attention output weight, bias
        out += [h, h]                           # attention LayerNorm gamma, beta
        out += [h * ff, ff]                     # FFN in weight, bias
        out += [ff * h, h]                      # FFN out weight, bias
        out += [h, h]                           # output LayerNorm gamma, beta
    return out


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    numel: tuple
    n_workers: int
    grad_dtype: int
    law: str                  # "iid", "block_sigma", "heavy_tail", "tensor_std"
    grad_std: float = 1e-3
    tensor_std: tuple = ()    # per-tensor standard deviations of the "tensor_std" law
    warmup_steps: int = 5
    compress_steps: int = 5
    seed: int = 0
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    lr: float = 1e-3
    param_std: float = 0.02

    @property
    def d(self) -> int:
        return int(sum(self.numel))

    @property
    def n_tensors(self) -> int:
        return len(self.numel)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", (1 << 20,), 4, F32, "iid", warmup_steps=5, compress_steps=5, seed=0),
    "bert_base": Workload("bert_base", (110_000_000,), 8, F32, "block_sigma", warmup_steps=100,
                          compress_steps=50, seed=1),
    "bert_large": Workload("bert_large", (340_000_000,), 16, F16, "block_sigma", warmup_steps=20,
                           compress_steps=50, seed=2),
    "ragged_bert_large": Workload("ragged_bert_large", tuple(bert_large_shapes()), 8, F32, "iid",
                                  warmup_steps=5, compress_steps=20, seed=3),
    "gpt2_1p5b": Workload("gpt2_1p5b", (1_560_000_000,), 4, BF16, "heavy_tail", warmup_steps=5,
                          compress_steps=20, seed=4),
    # one flat buffer past 2^31 elements: checks that no element index is held in 32 bits
    "over_2g": Workload("over_2g", (2_200_000_000,), 2, BF16, "iid", warmup_steps=2, compress_steps=2, seed=5),
}

BLOCK = 1 << 20


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & ((1 << 63) - 1))
    return g


def params(w: Workload, device="cpu") -> list[torch.Tensor]:
    """Initial parameters, one fp32 tensor per entry of ``w.numel``, ~ N(0, param_std^2)."""
    g = _gen(device, w.seed * 7919 + 17)
    return [torch.randn(int(k), generator=g, device=device, dtype=torch.float32) * w.param_std
            for k in w.numel]


def _block_sigma(w: Workload, device) -> torch.Tensor:
    nblk = max(1, math.ceil(w.d / BLOCK))
    g = _gen(device, w.seed * 104729 + 3)
    u = torch.rand(nblk, generator=g, device=device, dtype=torch.float64)
    return torch.pow(10.0, -5.0 + 3.0 * u).to(torch.float32)


def _heavy_mask(w: Workload, device) -> torch.Tensor:
    g = _gen(device, w.seed * 15485863 + 5)
    return torch.rand(w.d, generator=g, device=device) < 0.01


class GradSource:
    """Per-step gradients: ``grads(step)`` -> list of n*T tensors ordered [worker][tensor]."""

    def __init__(self, w: Workload, device="cpu"):
        self.w = w
        self.device = device
        self._sigma = _block_sigma(w, device) if w.law == "block_sigma" else None
        self._heavy = _heavy_mask(w, device) if w.law == "heavy_tail" else None

    def _flat(self, gen: torch.Generator) -> torch.Tensor:
        w = self.w
        z = torch.randn(w.d, generator=gen, device=self.device, dtype=torch.float32)
        if w.law == "iid":
            z.mul_(w.grad_std)
        elif w.law == "block_sigma":
            nfull = w.d // BLOCK
            if nfull:
                z[: nfull * BLOCK].view(nfull, BLOCK).mul_(self._sigma[:nfull, None])
            if w.d > nfull * BLOCK:
                z[nfull * BLOCK:].mul_(self._sigma[nfull])
        elif w.law == "heavy_tail":
            z.mul_(w.grad_std)
            z[self._heavy] *= 100.0
        elif w.law == "tensor_std":
            off = 0
            for L, sd in zip(w.numel, w.tensor_std):
                z[off: off + int(L)].mul_(sd)
                off += int(L)
        else:
            raise ValueError(w.law)
        return z.to(TORCH_DTYPE[w.grad_dtype])

    def grads(self, step: int) -> list[torch.Tensor]:
        w = self.w
        out = []
        for i in range(w.n_workers):
            gen = _gen(self.device, (w.seed * 1_000_003 + step) * 1031 + i)
            flat = self._flat(gen)
            out += list(torch.split(flat, list(w.numel)))
        return out


def to_numpy_grad(t: torch.Tensor):
    """Host copy of a gradient tensor in the form the oracle takes (bf16 as its uint16 bits)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
