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

  1. gradients   window by window ("【论文解读】ZeRO" sec. 4(2): gradients are reduced in
                 buckets at the partition boundaries): every process's range is cut on one
                 flat grid of w elements, and at exchange k each process receives its k-th
                 window from every other process (point-to-point sends of the flat slice
                 of each local gradient copy), so every process sends and receives alike;
                 the windows land in two constant-size receive slots (sec. 5(2),
                 constant-size buffers), and the exchanges of the next windows are in
                 flight while this one is reduced.  w is a multiple of the 8192-element
                 tile grid, so no tile of the sums of squares is split between windows and
                 the result does not depend on w;
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


def exchange_windows(local_len: int, world: int, w: int) -> list[list[tuple[int, int]]]:
    """For every process q, its flat range [q * local_len, (q + 1) * local_len) cut at the
    flat multiples of w: a list of (begin, count) in order.  w = 0: one window per range."""
    out = []
    for q in range(world):
        lo, hi = q * local_len, (q + 1) * local_len
        if w == 0:
            out.append([(lo, local_len)])
            continue
        ws, b = [], lo
        while b < hi:
            e = min((b // w + 1) * w, hi)
            ws.append((b, e - b))
            b = e
        out.append(ws)
    return out


def exchange_plan(windows, me: int, k: int, copies: int, part: int):
    """Exchange k for process `me`: sends (peer, local copy j, flat begin, count) of the
    peer's k-th window out of each local gradient copy, and receives (peer, local copy j,
    offset in the receive slot, count) of its own k-th window from every peer, at
    peer * part in copy j's slot.  Between two processes the messages are listed in the
    same order on both sides (by copy), which is how point-to-point messages match."""
    sends, recvs = [], []
    for q in range(len(windows)):
        if q == me:
            continue
        if k < len(windows[q]):
            b, n = windows[q][k]
            sends += [(q, j, b, n) for j in range(copies)]
        if k < len(windows[me]):
            _, n = windows[me][k]
            recvs += [(q, j, q * part, n) for j in range(copies)]
    return sends, recvs


class _Done:
    def wait(self) -> None:
        pass


class _Pending:
    """Exchanges in flight: wait() completes them (and, for host-staged tensors, copies
    the results into the device tensors)."""

    def __init__(self, works, copies=()):
        self.works, self.copies = list(works), list(copies)

    def wait(self) -> None:
        for w in self.works:
            if w is not None:
                w.wait()
        for dst, src in self.copies:
            dst.copy_(src)


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
            pend = _Pending([work], [(o, oh)])
        else:
            work = dist.all_to_all_single(o, i, output_split_sizes=os_, input_split_sizes=is_,
                                          group=self.group, async_op=async_op)
            pend = _Pending([work])
        if not async_op:
            pend.wait()
            return _Done()
        return pend

    def send_recv(self, sends, recvs):
        """Point-to-point: sends and recvs are lists of (peer, tensor); messages between
        two processes are matched in the order they are listed.  Asynchronous: returns a
        handle whose wait() completes them all."""
        ops, copies = [], []
        for peer, t in sends:
            b = t.view(torch.uint8)
            ops.append(dist.P2POp(dist.isend, b.cpu() if self._host(b) else b, peer, self.group))
        for peer, t in recvs:
            b = t.view(torch.uint8)
            if self._host(b):
                h = torch.empty(b.numel(), dtype=torch.uint8)
                copies.append((b, h))
                b = h
            ops.append(dist.P2POp(dist.irecv, b, peer, self.group))
        if not ops:
            return _Done()
        return _Pending(dist.batch_isend_irecv(ops), copies)

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

    layout          from zero_partition with align = 8 (the local buffers start at flat
                    origin = rank_begin * S, which must be a multiple of 8)
    dtype           ZERO_F16 or ZERO_BF16: the gradient copies' element type
    exchange_elems  w: the gradient exchange's window, a multiple of 8192 (the tile grid);
                    0 = each process's whole range at once.  The receive buffers hold
                    2 * world * w elements per local copy (world * range when w = 0).
                    The result does not depend on w.
    """

    def __init__(self, layout, hp, dtype: int, loss_scale: float = 1.0, dynamic: bool = False,
                 growth_interval: int = 1000, device=None, group=None, exchange_elems: int = 0):
        if exchange_elems < 0 or exchange_elems % 8192:
            raise ValueError("exchange_elems must be a multiple of 8192 (or 0)")
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
        self.windows_of = exchange_windows(self.local_len, self.world, exchange_elems)
        self.n_exchanges = max(len(w) for w in self.windows_of)
        # every rank's copy of one window of this process's range arrives here: per local
        # copy and slot (two slots: the next windows' exchanges overlap this window's
        # reduce), world * w elements, process q's part at q * w
        self.slots = 2 if self.n_exchanges > 1 else 1
        w_max = max((n for ws in self.windows_of for _, n in ws), default=0)
        self.part = w_max
        self.recv = [[torch.empty(self.world * w_max, dtype=torch.int16, device=dev)
                      for _ in range(self.rank_count)] for _ in range(self.slots)] \
            if self.world > 1 else []
        zero_step_state_init(layout, loss_scale, dynamic, growth_interval, self.st, self.partials)

    def windows(self) -> list[tuple[int, int]]:
        """This process's reduce windows (begin, count), in order."""
        return self.windows_of[self.proc]

    def _issue(self, k: int, copies: Sequence[torch.Tensor]):
        """Exchange k: send every other process its k-th window of each local copy, and
        receive this process's k-th window of every other process's copies."""
        recv = self.recv[k % self.slots]
        sends, recvs = exchange_plan(self.windows_of, self.proc, k, self.rank_count, self.part)
        return self.ex.send_recv([(q, copies[j][b:b + n]) for q, j, b, n in sends],
                                 [(q, recv[j][o:o + n]) for q, j, o, n in recvs])

    def _sources(self, k: int, copies: Sequence[torch.Tensor]) -> list[int]:
        """Device address, for rank i = 0 .. N-1, of the first element of this process's
        window k in rank i's copy."""
        b, _ = self.windows_of[self.proc][k]
        R = self.rank_count
        recv = self.recv[k % self.slots] if self.world > 1 else None
        out = []
        for i in range(self.lay.n_ranks):
            q, j = divmod(i, R)
            if q == self.proc:
                out.append(copies[j].data_ptr() + 2 * b)
            else:
                out.append(recv[j].data_ptr() + 2 * q * self.part)
        return out

    def step(self, copies: Sequence[torch.Tensor], mark=None) -> None:
        """One optimizer step on the current stream (the one torch.distributed orders its
        collectives against).  copies: this process's rank_count gradient copies (ranks
        rank_begin, rank_begin+1, ... in order), psi_padded 16-bit elements each, on the
        device; their padding elements are ignored.  mark: optional callable, called with
        the name of each part as it has been enqueued ("gradients", "norm inputs",
        "norm", "adamw", "parameters"; "gradients" is the exchange and the reduce of every
        window, which overlap), e.g. to record timing events."""
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
        # 1. window by window: every rank's copy of this process's window arrives, then the
        #    reduce; exchange k+2 reuses k's slot once k's reduce is enqueued (a collective
        #    is ordered after the work already on the stream)
        K = self.n_exchanges
        mine = self.windows_of[self.proc]
        pending = {}
        if self.world > 1:
            for k in range(min(self.slots, K)):
                pending[k] = self._issue(k, copies)
        for k in range(K):
            if k in pending:
                pending.pop(k).wait()
            if k < len(mine):
                begin, n = mine[k]
                zero_reduce_shard_unscale_local(lay, self.dtype, self.rank_begin, R,
                                                self._sources(k, copies), begin, n, self.g,
                                                self.partials, self.st, s)
            if self.world > 1 and k + self.slots < K:
                pending[k + self.slots] = self._issue(k + self.slots, copies)
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


__all__ = ["Exchange", "RankStep", "local_ranks", "layout_for", "exchange_windows",
           "exchange_plan", "OVERFLOW_WORD"]
