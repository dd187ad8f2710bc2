"""The ZeRO step with its ranks spread over processes (one process per GPU).

"【论文解读】ZeRO" sec. 6(2) and the stage-2 flow of "ZeRO技术概述": every rank receives each
rank's gradient of its own partition (the reduce-scatter), updates only that partition of
the fp32 optimizer state, and the updated parameters are all-gathered.  The Megatron
distributed-optimizer page (sec. 1): one all-reduce forms the global gradient norm before
clipping.  Here each process holds a contiguous group of the N ranks, [rank_begin,
rank_begin + rank_count), and only their part of g, master, m and v.

Every step of the arithmetic runs in the library's kernels, through the C ABI:
zero_reduce_shard_unscale_local, zero_grad_norm and zero_adamw_cast_gather_local.  This
module only moves data between processes with torch.distributed (NCCL on the device
buffers; gloo through host memory):

  1. gradients   bucket by bucket (the layout's bucket grid, "【论文解读】ZeRO" sec. 4(2):
                 gradients are reduced in buckets at the partition boundaries), one
                 all-to-all per local gradient copy: the bucket's flat slice of a copy
                 already lies in destination order, since every process's range is
                 contiguous, so it is sent as it is with one split per process, and each
                 process receives every rank's copy of its part of the bucket into a
                 constant-size buffer (sec. 5(2), constant-size buffers); the exchange of
                 the next bucket is issued before this bucket's reduce;
  2. norm        all-gather of every process's tile partials (fp64, a few bytes per 8192
                 parameters) and a maximum over processes of the step state's overflow
                 word; each process then forms the same norm, clip coefficient, scaler
                 update and skip decision;
  3. parameters  all-gather of each process's 16-bit parameters into the full buffer.

The reduce-scatter is an all-to-all of the raw 16-bit copies followed by the local fp32 sum
in ascending rank order, rather than NCCL's reduce-scatter: each process sends and receives
the same (G-1)/G of its copies either way, but the order of the sum is then fixed, so
every output equals the one-GPU step's (zero_step on the same layout) bit for bit, wherever
the ranks live.  16-bit buffers travel as bytes (gloo has no 16-bit integer type).
"""
from __future__ import annotations

from typing import Sequence

import torch
import torch.distributed as dist

from . import (STATE_BYTES, StepState, zero_adamw_cast_gather_local, zero_grad_norm,
               zero_partition, zero_reduce_shard_unscale_local, zero_step_state_init)

# index of the step state's overflow word in an int32 view of the 128-byte state
OVERFLOW_WORD = StepState.overflow.offset // 4


def local_ranks(n_ranks: int, world: int, proc: int) -> tuple[int, int]:
    """(rank_begin, rank_count): the contiguous ranks process `proc` of `world` holds."""
    if world < 1 or not 0 <= proc < world or n_ranks % world:
        raise ValueError(f"{n_ranks} ranks cannot be split evenly over {world} processes")
    count = n_ranks // world
    return proc * count, count


class _Done:
    def wait(self) -> None:
        pass


class _Pending:
    """An exchange in flight: wait() completes it (and, for host-staged tensors, copies the
    result into the device tensor)."""

    def __init__(self, work, out=None, host=None):
        self.work, self.out, self.host = work, out, host

    def wait(self) -> None:
        if self.work is not None:
            self.work.wait()
        if self.host is not None:
            self.out.copy_(self.host)


class Exchange:
    """The step's collectives over torch.distributed, on tensors of any device.

    With NCCL the collectives run on the device tensors themselves, ordered after the
    work already enqueued on the current stream, and wait() makes the current stream wait
    for them.  With another backend (gloo), device tensors are copied to host memory,
    exchanged there and copied back; host tensors are exchanged directly.
    """

    def __init__(self, group=None):
        self.group = group
        self.world = dist.get_world_size(group)
        self.proc = dist.get_rank(group)
        self.nccl = dist.get_backend(group) == "nccl"

    def _host(self, t: torch.Tensor) -> bool:
        return t.is_cuda and not self.nccl

    def all_to_all(self, out: torch.Tensor, inp: torch.Tensor, out_splits=None, in_splits=None,
                   async_op: bool = False):
        """Part q of `inp` goes to process q; part q of `out` comes from process q.  Parts
        are equal unless split sizes (in elements of the tensors' type) are given.  Returns
        a handle whose wait() completes the exchange (already complete unless async_op)."""
        o, i = out.view(torch.uint8), inp.view(torch.uint8)
        k = out.element_size()
        os_ = None if out_splits is None else [k * x for x in out_splits]
        is_ = None if in_splits is None else [k * x for x in in_splits]
        if self._host(o):
            oh = torch.empty(o.numel(), dtype=torch.uint8)
            work = dist.all_to_all_single(oh, i.cpu(), output_split_sizes=os_, input_split_sizes=is_,
                                          group=self.group, async_op=async_op)
            pend = _Pending(work, o, oh)
        else:
            work = dist.all_to_all_single(o, i, output_split_sizes=os_, input_split_sizes=is_,
                                          group=self.group, async_op=async_op)
            pend = _Pending(work)
        if not async_op:
            pend.wait()
            return _Done()
        return pend

    def all_gather(self, full: torch.Tensor, lo: int, hi: int) -> None:
        """Every process contributes full[lo:hi] (its own part, the same length on each);
        afterwards `full` holds all parts in process order."""
        part = full[lo:hi]
        if full.dtype in (torch.int16, torch.float16, torch.bfloat16):
            full, part = full.view(torch.uint8), part.view(torch.uint8)
        if self._host(full):
            fh = torch.empty(full.numel(), dtype=full.dtype)
            dist.all_gather_into_tensor(fh, part.cpu(), group=self.group)
            full.copy_(fh)
        else:
            # the input is a copy of this process's part, never a view into the output
            dist.all_gather_into_tensor(full, part.clone(), group=self.group)

    def maximum(self, t: torch.Tensor) -> None:
        """Element-wise maximum over processes, in place."""
        if self._host(t):
            th = t.cpu()
            dist.all_reduce(th, op=dist.ReduceOp.MAX, group=self.group)
            t.copy_(th)
        else:
            dist.all_reduce(t, op=dist.ReduceOp.MAX, group=self.group)


class RankStep:
    """One process's part of the ZeRO step: its ranks' g, master, m, v (local_len =
    rank_count * S elements each, flat index - origin), the full gathered parameters, the
    full tile partials and the step state, all on `device`.  The state arrays start at 0;
    fill them (e.g. from a checkpoint) before the first step.

    layout      from zero_partition with align = 8 (the local buffers start at flat
                origin = rank_begin * S, which must be a multiple of 8); its bucket size
                sets the gradient exchange's granularity and the receive buffers' size
    dtype       ZERO_F16 or ZERO_BF16: the gradient copies' element type
    """

    def __init__(self, layout, hp, dtype: int, loss_scale: float = 1.0, dynamic: bool = False,
                 growth_interval: int = 1000, device=None, group=None):
        self.lay, self.hp, self.dtype = layout, hp, dtype
        self.ex = Exchange(group)
        self.world, self.proc = self.ex.world, self.ex.proc
        self.rank_begin, self.rank_count = local_ranks(layout.n_ranks, self.world, self.proc)
        S, P = layout.shard, layout.psi_padded
        self.origin, self.local_len = self.rank_begin * S, self.rank_count * S
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.dev = dev
        self.g = torch.empty(self.local_len, dtype=torch.float32, device=dev)
        self.master = torch.zeros(self.local_len, dtype=torch.float32, device=dev)
        self.m = torch.zeros(self.local_len, dtype=torch.float32, device=dev)
        self.v = torch.zeros(self.local_len, dtype=torch.float32, device=dev)
        self.params = torch.zeros(P, dtype=torch.int16, device=dev)
        self.params_local = self.params[self.origin:self.origin + self.local_len]
        self.partials = torch.empty(layout.n_tiles, dtype=torch.float64, device=dev)
        self.st = torch.empty(STATE_BYTES, dtype=torch.uint8, device=dev)
        self.buckets = self._buckets()
        # every rank's copy of this process's part of a bucket arrives here: one buffer per
        # local copy and slot (two slots: the next bucket's exchange overlaps this bucket's
        # reduce), world * (this process's largest part of a bucket) elements each
        self.slots = 2 if len(self.buckets) > 1 else 1
        part = max(sizes[self.proc] for _, _, sizes in self.buckets)
        self.recv = [[torch.empty(self.world * part, dtype=torch.int16, device=dev)
                      for _ in range(self.rank_count)] for _ in range(self.slots)] \
            if self.world > 1 else []
        zero_step_state_init(layout, loss_scale, dynamic, growth_interval, self.st, self.partials)

    def _buckets(self) -> list[tuple[int, int, list[int]]]:
        """(lo, hi, sizes) per bucket of the layout's grid: sizes[q] is the part of
        [lo, hi) inside process q's range (the ranges are contiguous and in order, so the
        parts follow each other)."""
        W, P, L = self.lay.bucket_elems, self.lay.psi_padded, self.local_len
        out = []
        for b in range(self.lay.n_buckets):
            lo, hi = b * W, min((b + 1) * W, P)
            sizes = [max(0, min(hi, (q + 1) * L) - max(lo, q * L)) for q in range(self.world)]
            out.append((lo, hi, sizes))
        return out

    def windows(self) -> list[tuple[int, int]]:
        """The layout's reduce windows (its bucket grid) clipped to the local range."""
        lo_r = self.origin
        return [(max(lo, lo_r), sizes[self.proc]) for lo, _, sizes in self.buckets
                if sizes[self.proc] > 0]

    def _issue(self, b: int, copies: Sequence[torch.Tensor]) -> list:
        lo, hi, sizes = self.buckets[b]
        n = sizes[self.proc]
        recv = self.recv[b % self.slots]
        return [self.ex.all_to_all(recv[j][:self.world * n], copies[j][lo:hi],
                                   out_splits=[n] * self.world, in_splits=sizes, async_op=True)
                for j in range(self.rank_count)]

    def _sources(self, b: int, copies: Sequence[torch.Tensor]) -> list[int]:
        """Device address, for rank k = 0 .. N-1, of the first element of this process's
        part of bucket b in rank k's copy."""
        lo, _, sizes = self.buckets[b]
        R, n = self.rank_count, sizes[self.proc]
        begin = max(lo, self.origin)
        recv = self.recv[b % self.slots] if self.world > 1 else None
        out = []
        for k in range(self.lay.n_ranks):
            q, j = divmod(k, R)
            if q == self.proc:
                out.append(copies[j].data_ptr() + 2 * begin)
            else:
                out.append(recv[j].data_ptr() + 2 * q * n)
        return out

    def step(self, copies: Sequence[torch.Tensor], mark=None) -> None:
        """One optimizer step on the current stream (the one torch.distributed orders its
        collectives against).  copies: this process's rank_count gradient copies (ranks
        rank_begin, rank_begin+1, ... in order), psi_padded 16-bit elements each, on the
        device; their padding elements are ignored.  mark: optional callable, called with
        the name of each part as it has been enqueued ("gradients", "norm inputs",
        "norm", "adamw", "parameters"; "gradients" is the exchange and the reduce of every
        bucket, which overlap), e.g. to record timing events."""
        lay, R = self.lay, self.rank_count
        if len(copies) != R:
            raise ValueError(f"expected {R} gradient copies, got {len(copies)}")
        for c in copies:  # the kernels read them through raw addresses: check before
            if (not c.is_cuda or c.device != self.dev or c.element_size() != 2
                    or c.numel() != lay.psi_padded or not c.is_contiguous()):
                raise ValueError("each gradient copy must be a contiguous 16-bit tensor of "
                                 f"psi_padded = {lay.psi_padded} elements on {self.dev}")
        s = torch.cuda.current_stream(self.dev)
        mark = mark or (lambda name: None)
        # 1. bucket by bucket: every rank's copy of this process's part arrives, then the
        #    reduce; bucket b+2's exchange reuses b's slot once b's reduce is enqueued (the
        #    exchange is ordered after the work already on the stream)
        nb = len(self.buckets)
        pending = {}
        if self.world > 1:
            for b in range(min(self.slots, nb)):
                pending[b] = self._issue(b, copies)
        for b in range(nb):
            for h in pending.pop(b, []):
                h.wait()
            lo, _, sizes = self.buckets[b]
            n = sizes[self.proc]
            if n > 0:
                zero_reduce_shard_unscale_local(lay, self.dtype, self.rank_begin, R,
                                                self._sources(b, copies), max(lo, self.origin),
                                                n, self.g, self.partials, self.st, s)
            if self.world > 1 and b + self.slots < nb:
                pending[b + self.slots] = self._issue(b + self.slots, copies)
        mark("gradients")
        # 2. the global norm's inputs: every process's tile partials and overflow flag
        if self.world > 1:
            tpr = lay.tiles_per_rank
            self.ex.all_gather(self.partials, self.rank_begin * tpr, (self.rank_begin + R) * tpr)
            self.ex.maximum(self.st.view(torch.int32)[OVERFLOW_WORD:OVERFLOW_WORD + 1])
        mark("norm inputs")
        zero_grad_norm(lay, self.hp, self.partials, self.st, s)
        mark("norm")
        # 3. this process's shards, then the parameter all-gather
        zero_adamw_cast_gather_local(lay, self.hp, self.rank_begin, R, self.g, self.master,
                                     self.m, self.v, self.params_local, self.st, s)
        mark("adamw")
        if self.world > 1:
            self.ex.all_gather(self.params, self.origin, self.origin + self.local_len)
        mark("parameters")


def layout_for(psi: int, n_ranks: int, stage: int = 2, bucket_elems: int = 0):
    """zero_partition with the alignment rank-local buffers need (S a multiple of 8)."""
    return zero_partition(psi, n_ranks, stage, 8, bucket_elems)


__all__ = ["Exchange", "RankStep", "local_ranks", "layout_for", "OVERFLOW_WORD"]
