"""Multi-GPU form of the 1-bit Adam step: one process per GPU, the n workers spread over the ranks.

The pages' system exchanges the compressed momenta across machines ("1-bit Adam: Communication
Efficient Large-Scale Training with Adam's Convergence Speed", Sec. 6 and Sec. 11 steps 1-3): every
worker compresses its momentum with error compensation, an all-to-all gives each server the workers'
compressed chunks of its shard, every server averages them, compresses again with its own error, and
an all-gather brings the servers' results to every worker, which updates its copy of the model (the
AIMech page's "gather-then-broadcast"; the 1-bit LAMB page's abstract runs this over NCCL).

Here rank r of ``world`` simulates workers r*nl .. r*nl+nl-1 (nl = n/world) and serves the same
numbered shards of every tensor.  The compute is the library's: ``onebit_adam_compress_begin`` (worker
kernel + packing), ``onebit_adam_compress_serve`` (unpacking, server kernel, packing of this rank's
result) and ``onebit_adam_compress_end`` (unpacking of the broadcast, update); see
``include/onebit_adam.h``.  This module only allocates the exchange buffers and moves them with
``torch.distributed`` collectives between those calls.  Results are bit-identical to one GPU
simulating all n workers.

Transports (how the buffers travel):
  * ``DeviceTransport``: collectives on the device buffers (NCCL process groups);
  * ``HostTransport``: the buffers staged through host memory (gloo process groups, for example
    several ranks sharing one GPU in a test);
  * ``LocalTransport``: one rank, nothing to move.
"""
from __future__ import annotations

import contextlib
import ctypes

import torch
import torch.distributed as tdist

from . import OK, PHASE_WARMUP, OneBitAdam, _check, _stream_ptr, lib


def _bind(L):
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sig = {
        "onebit_adam_workspace_size_rank": [vp, i32, i32, ctypes.POINTER(ctypes.c_size_t)],
        "onebit_adam_init_rank": [vp, i32, i32, ctypes.POINTER(vp), vp, ctypes.c_size_t, vp, ctypes.POINTER(vp)],
        "onebit_adam_exchange_words": [vp, ctypes.POINTER(i64), ctypes.POINTER(i64)],
        "onebit_adam_compress_begin": [vp, ctypes.POINTER(vp), vp, vp],
        "onebit_adam_compress_serve": [vp, vp, vp, vp],
        "onebit_adam_compress_end": [vp, vp, vp],
        "onebit_adam_plan_exchange": [vp, i32, i32, ctypes.POINTER(i64), i64, ctypes.POINTER(i64),
                                      ctypes.POINTER(i64), ctypes.POINTER(i64)],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    return L


def _lib():
    L = lib()
    if not getattr(L, "_dist_bound", False):
        _bind(L)
        L._dist_bound = True
    return L


def plan_exchange(cfg, rank: int, world: int):
    """The exchange copies of rank `rank` of `world` (host only): (rows, send_block, bcast_block), rows
    being tuples (stage, src region, src row, src offset, dst region, dst row, dst offset, words)."""
    count, sb, bb = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    L = _lib()
    _check(L.onebit_adam_plan_exchange(ctypes.byref(cfg), rank, world, None, 0, ctypes.byref(count), ctypes.byref(sb),
                                       ctypes.byref(bb)), "onebit_adam_plan_exchange")
    rows = (ctypes.c_int64 * (8 * max(count.value, 1)))()
    _check(L.onebit_adam_plan_exchange(ctypes.byref(cfg), rank, world, rows, count.value, ctypes.byref(count),
                                       ctypes.byref(sb), ctypes.byref(bb)), "onebit_adam_plan_exchange")
    return [tuple(rows[8 * q: 8 * q + 8]) for q in range(count.value)], sb.value, bb.value


def workspace_size_rank(cfg, rank: int, world: int) -> int:
    out = ctypes.c_size_t()
    _check(_lib().onebit_adam_workspace_size_rank(ctypes.byref(cfg), rank, world, ctypes.byref(out)),
           "onebit_adam_workspace_size_rank")
    return out.value


# ---------------------------------------------------------------------------------- transports

class LocalTransport:
    """One rank: nothing to move (the library does not touch the buffers when world == 1)."""

    def all_to_all(self, recv, send):
        pass

    def all_gather(self, gathered, block):
        pass

    def all_gather_flat(self, out, local):
        out.copy_(local)


class DeviceTransport:
    """Collectives on the device buffers themselves (an NCCL process group)."""

    def __init__(self, group=None):
        self.group = group

    def all_to_all(self, recv, send):
        tdist.all_to_all_single(recv, send, group=self.group)

    def all_gather(self, gathered, block):
        tdist.all_gather_into_tensor(gathered, block, group=self.group)

    def all_gather_flat(self, out, local):
        tdist.all_gather_into_tensor(out, local, group=self.group)


class HostTransport:
    """The buffers staged through host memory around CPU collectives (a gloo process group)."""

    def __init__(self, group=None):
        self.group = group

    def _gather(self, out_cpu, block_cpu):
        try:
            tdist.all_gather_into_tensor(out_cpu, block_cpu, group=self.group)
        except (RuntimeError, NotImplementedError):  # older gloo builds: the list form
            world = tdist.get_world_size(self.group)
            tdist.all_gather(list(out_cpu.view(world, -1).unbind(0)), block_cpu, group=self.group)

    def all_to_all(self, recv, send):
        r = torch.empty(recv.shape, dtype=recv.dtype)
        tdist.all_to_all_single(r, send.cpu(), group=self.group)
        recv.copy_(r)

    def all_gather(self, gathered, block):
        g = torch.empty(gathered.shape, dtype=gathered.dtype)
        self._gather(g, block.cpu())
        gathered.copy_(g)

    def all_gather_flat(self, out, local):
        g = torch.empty(out.shape, dtype=out.dtype)
        self._gather(g, local.cpu())
        out.copy_(g)


# ---------------------------------------------------------------------------------- the rank optimizer

class ExchangeError(RuntimeError):
    """A collective of a compression step failed; the step was abandoned (see RankOneBitAdam)."""


class RankOneBitAdam(OneBitAdam):
    """Rank `rank` of `world` of the multi-GPU 1-bit Adam step (n_workers a multiple of world).

    ``warmup_step(local_grads)`` and ``compress_step(local_grads)`` take this rank's nl*T gradient
    tensors ([local worker][tensor]); every other method is the single-GPU handle's.  The warm-up's
    uncompressed exchange is an all-gather of the ranks' gradients, after which every rank computes
    the same ordered mean of all n (bit-identical to one GPU; a ring all-reduce would reorder the fp32
    sum).
    """

    def __init__(self, params, n_workers, warmup_steps, rank, world, transport=None, beta1=0.9, beta2=0.999,
                 eps=1e-8, lr=1e-3, grad_dtype=None, bias_correction=False, workspace=None, stream=None,
                 scale_block=0):
        from . import F32, _torch_dtype_code, make_config

        self.params = list(params)
        for p in self.params:
            if p.dtype != torch.float32 or not p.is_cuda or not p.is_contiguous():
                raise ValueError("parameters must be contiguous fp32 CUDA tensors")
        self.n = int(n_workers)
        self.rank, self.world = int(rank), int(world)
        if self.world < 1 or not 0 <= self.rank < self.world or self.n % self.world:
            raise ValueError("need 0 <= rank < world and n_workers a multiple of world")
        self.nl = self.n // self.world
        self.T = len(self.params)
        self.numel = [p.numel() for p in self.params]
        gdt = F32 if grad_dtype is None else (grad_dtype if isinstance(grad_dtype, int) else _torch_dtype_code(grad_dtype))
        self.grad_dtype = gdt
        self.cfg = make_config(self.numel, self.n, warmup_steps, beta1, beta2, eps, lr, gdt, bias_correction,
                               scale_block)
        self.workspace = workspace
        self.transport = transport if transport is not None else (LocalTransport() if self.world == 1 else
                                                                   DeviceTransport())
        L = _lib()
        ptrs = (ctypes.c_void_p * self.T)(*[p.data_ptr() for p in self.params])
        h = ctypes.c_void_p()
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        _check(L.onebit_adam_init_rank(ctypes.byref(self.cfg), self.rank, self.world, ptrs, ws_ptr, ws_bytes,
                                       _stream_ptr(stream), ctypes.byref(h)), "onebit_adam_init_rank")
        self.h = h
        sb, bb = ctypes.c_int64(), ctypes.c_int64()
        _check(L.onebit_adam_exchange_words(self.h, ctypes.byref(sb), ctypes.byref(bb)), "onebit_adam_exchange_words")
        self.send_block, self.bcast_block = sb.value, bb.value
        dev = self.params[0].device
        w = self.world if self.world > 1 else 0  # one rank moves nothing
        self.send = torch.empty(w * self.send_block, dtype=torch.int32, device=dev)
        self.recv = torch.empty(w * self.send_block, dtype=torch.int32, device=dev)
        self.bcast = torch.empty(self.bcast_block if w else 0, dtype=torch.int32, device=dev)
        self.gathered = torch.empty(w * self.bcast_block, dtype=torch.int32, device=dev)

    def _ptr(self, t):
        return t.data_ptr() if t.numel() else None

    def _local_grad_array(self, grads):
        return self._grad_array(grads, count=self.nl * self.T)

    def all_gradients(self, local_grads):
        """Every worker's gradients ([worker][tensor], n*T tensors) from each rank's nl*T: the warm-up's
        uncompressed exchange, as an all-gather."""
        if len(local_grads) != self.nl * self.T:
            raise ValueError(f"expected {self.nl * self.T} local gradient tensors, got {len(local_grads)}")
        if self.world == 1:
            return list(local_grads)
        local = torch.cat([g.reshape(-1) for g in local_grads])
        out = torch.empty(self.world * local.numel(), dtype=local.dtype, device=local.device)
        self.transport.all_gather_flat(out, local)
        return list(torch.split(out, self.numel * self.n))

    def warmup_step(self, local_grads, stream=None):
        with torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext():
            super().warmup_step(self.all_gradients(local_grads), stream)

    # the three library calls of a compression step; compress_step() runs them with the collectives
    def begin(self, local_grads, stream=None):
        """Worker step: fills self.send (block q: this rank's messages for rank q's shards)."""
        _check(_lib().onebit_adam_compress_begin(self.h, self._local_grad_array(local_grads), self._ptr(self.send),
                                                 _stream_ptr(stream)), "onebit_adam_compress_begin", self.h)

    def serve(self, stream=None):
        """Server step on self.recv (block p: rank p's messages for this rank's shards); fills self.bcast."""
        _check(_lib().onebit_adam_compress_serve(self.h, self._ptr(self.recv), self._ptr(self.bcast),
                                                 _stream_ptr(stream)), "onebit_adam_compress_serve", self.h)

    def end(self, stream=None):
        """Broadcast and update from self.gathered (every rank's bcast block, in rank order)."""
        _check(_lib().onebit_adam_compress_end(self.h, self._ptr(self.gathered), _stream_ptr(stream)),
               "onebit_adam_compress_end", self.h)

    def compress_step(self, local_grads, stream=None):
        # the collectives run on the same stream as the library's kernels, so that they are ordered
        with torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext():
            self.begin(local_grads, stream)
            try:
                self.transport.all_to_all(self.recv, self.send)
                self.serve(stream)
                self.transport.all_gather(self.gathered, self.bcast)
            except Exception as e:  # a peer failed or left: leave the split step, report, keep the handle usable
                t, phase = self.get_step()
                self.set_step(t, phase, stream)
                raise ExchangeError(f"rank {self.rank} of {self.world}: the exchange of compression step {t + 1} "
                                    f"failed ({e}); the step was abandoned and the optimizer state is not "
                                    "meaningful: restore it with load_state_dict()") from e
            self.end(stream)

    # ---- checkpoints: this rank's share of the state
    def state_dict(self, stream=None):
        """The step count and phase, m, v (den after the freeze), the errors of this rank's workers and
        the server error of its shards (other elements 0), as fp32 CUDA tensors."""
        from . import STATE_M, STATE_SERVER_ERROR, STATE_V, STATE_WORKER_ERROR

        t, phase = self.get_step()
        return {"t": t, "phase": phase, "rank": self.rank, "world": self.world,
                "m": self.export_state(STATE_M, stream=stream), "v": self.export_state(STATE_V, stream=stream),
                "server_error": self.export_state(STATE_SERVER_ERROR, stream=stream),
                "worker_error": {i: self.export_state(STATE_WORKER_ERROR, i, stream=stream)
                                 for i in range(self.rank * self.nl, (self.rank + 1) * self.nl)}}

    def load_state_dict(self, d, stream=None):
        """Restore a state_dict() taken on the same rank of the same configuration."""
        from . import STATE_M, STATE_SERVER_ERROR, STATE_V, STATE_WORKER_ERROR

        if (d.get("rank"), d.get("world")) != (self.rank, self.world):
            raise ValueError("the checkpoint belongs to another rank or world size")
        self.set_step(d["t"], d["phase"], stream=stream)
        self.import_state(STATE_M, d["m"], stream=stream)
        self.import_state(STATE_V, d["v"], stream=stream)
        self.import_state(STATE_SERVER_ERROR, d["server_error"], stream=stream)
        for i, e in d["worker_error"].items():
            self.import_state(STATE_WORKER_ERROR, e, int(i), stream=stream)

    def exchange_bytes(self):
        """Bytes this rank sends per compression step: all-to-all blocks to the other ranks, then its
        all-gather block to each of them."""
        w = self.world
        return 4 * (w - 1) * (self.send_block + self.bcast_block)


__all__ = ["RankOneBitAdam", "ExchangeError", "DeviceTransport", "HostTransport", "LocalTransport", "plan_exchange",
           "workspace_size_rank", "OK", "PHASE_WARMUP"]
