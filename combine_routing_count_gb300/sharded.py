"""Expert parallelism over several GPUs: the N expert-parallel ranks split into windows of
consecutive ranks, one window per process (one GPU each).

"Enabling trillion-parameter models on AWS EFA" (Perplexity), section "Send and receive
buffers": the routing information is exchanged first, so that every rank knows at which
offsets its writes land and where it receives from each rank; each rank then writes one
contiguous slice per peer. Section "MoE all-to-all over EFA": inside a node the slices go
over NVLink straight into the peers' buffers. Combine moves the same slices back.

A pass of one window (ShardedEP), in order:
  1. routing exchange: every window's expert ids [n, T, R] are all-gathered, and every
     process runs the same moe_layout on all N ranks' ids, so all layouts agree bit for bit;
  2. the exchange plan: moe_exchange_plan lists, from the layout's counts and offsets, the
     slices this window sends to and receives from every other window, in (s, d) order on
     both sides;
  3. dispatch send on the window (moe_dispatch_send / moe_quantize_dispatch_send with the
     layout's rank window): its tokens packed, and the slices inside the window written by
     the kernels;
  4. the dispatch exchange: each remote slice of the send buffer goes to its owner's
     receive buffer, one message per (s, d) slice;
  5. dispatch receive, identity expert and combine send on the window (the slices of
     sources inside the window written back by the kernels);
  6. the combine exchange: each remote slice of the combine-send buffer goes back to its
     source's combine-receive buffer;
  7. combine receive on the window: the weighted sum of every token's R rows.
Every row movement inside a window, and every computation, runs in libmoe_ep's kernels; the
transports only move whole contiguous slices between windows.

Transports: DistTransport uses a torch.distributed process group (NCCL between GPUs, gloo
for CPU tensors), one window per process; LocalTransport moves slices between several
windows held by one process (plain device copies), which runs the sharded pass of G windows
on one GPU.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from ._abi import (MOE_FLAG_DIRECT_PUSH, MOE_PAYLOAD_BF16, MOE_PAYLOAD_FP8_E4M3_B128, MoeDims, MoeLayout, MoeSlice,
                   check, lib)

__all__ = ["window_bounds", "exchange_plan", "ShardedEP", "DistTransport", "LocalTransport", "sharded_forward"]


def window_bounds(N: int, G: int) -> list[int]:
    """Rank windows of N ranks over G processes: window g holds ranks [b[g], b[g+1])."""
    if G < 1 or G > N:
        raise ValueError(f"cannot split {N} ranks into {G} windows")
    return [g * N // G for g in range(G + 1)]


def exchange_plan(dims: MoeDims, C: np.ndarray, soff: np.ndarray, roff: np.ndarray, bounds, me: int,
                  direction: int, sending: int) -> list[tuple[int, int, int, int, int]]:
    """moe_exchange_plan: the slices window `me` sends (sending=1) or receives (sending=0) in
    the dispatch (direction=0) or combine (direction=1) exchange, as (peer, s, d, rows,
    local_row) in ascending (s, d) order. C, soff, roff are host int32 arrays of the layout."""
    L = lib()
    C = np.ascontiguousarray(C, dtype=np.int32)
    soff = np.ascontiguousarray(soff, dtype=np.int32)
    roff = np.ascontiguousarray(roff, dtype=np.int32)
    b = np.ascontiguousarray(bounds, dtype=np.int32)
    args = (ctypes.byref(dims), C.ctypes.data, soff.ctypes.data, roff.ctypes.data, len(b) - 1, b.ctypes.data, int(me),
            int(direction), int(sending))
    n = L.moe_exchange_plan(*args, None, 0)
    if n < 0:
        raise ValueError("moe_exchange_plan: bad arguments")
    out = (MoeSlice * max(1, n))()
    got = L.moe_exchange_plan(*args, out, n)
    assert got == n
    return [(out[i].peer, out[i].s, out[i].d, out[i].rows, out[i].local_row) for i in range(n)]


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class ShardedEP:
    """One window [lo, hi) of an N-rank expert-parallel group: its ranks' buffers (window-local,
    rank lo + i in block i) and a layout of the whole group restricted to the window."""

    def __init__(self, N, T, H, E, R, cap=0, payload="bf16", *, bounds, me, flags=0):
        L_ = lib()
        self.fp8 = payload == "fp8"
        self.dims = MoeDims(N, T, H, E, R, cap, MOE_PAYLOAD_FP8_E4M3_B128 if self.fp8 else MOE_PAYLOAD_BF16)
        check(L_.moe_check_dims(ctypes.byref(self.dims)), "moe_check_dims")
        if flags & MOE_FLAG_DIRECT_PUSH:
            raise ValueError("direct push writes other windows' rows: not with a rank window")
        self.bounds = list(bounds)
        self.me = me
        self.lo, self.hi = self.bounds[me], self.bounds[me + 1]
        n = self.n = self.hi - self.lo
        self.N, self.T, self.H, self.E, self.R, self.L = N, T, H, E, R, E // N
        self.cap = L_.moe_capacity(ctypes.byref(self.dims))
        self.RB = L_.moe_recv_capacity_rows(ctypes.byref(self.dims))
        self.B = L_.moe_row_bytes(ctypes.byref(self.dims))
        dev = torch.device("cuda", torch.cuda.current_device())
        u8, bf16 = torch.uint8, torch.bfloat16
        ws = L_.moe_layout_workspace_bytes(ctypes.byref(self.dims))
        self.workspace = torch.empty(ws, dtype=u8, device=dev)
        self.layout = MoeLayout()
        check(L_.moe_layout_init(ctypes.byref(self.dims), self.workspace.data_ptr(), ws, ctypes.byref(self.layout),
                                 _stream()), "moe_layout_init")
        self.layout.flags = flags
        self.layout.win_lo, self.layout.win_hi = self.lo, self.hi
        Lx = self.L
        self.idx = torch.empty((N, T, R), dtype=torch.int32, device=dev)   # every rank's ids
        self.send = torch.empty((n, T * R, self.B), dtype=u8, device=dev)
        self.recv = torch.empty((n, self.RB, self.B), dtype=u8, device=dev)
        if self.fp8:
            self.expert_x = torch.empty((n, Lx, self.cap, H), dtype=u8, device=dev)
            self.expert_scale = torch.empty((n, Lx, self.cap, H // 128), dtype=torch.float32, device=dev)
            self.expert_y = torch.empty((n, Lx, self.cap, H), dtype=bf16, device=dev)
        else:
            self.expert_x = torch.empty((n, Lx, self.cap, H), dtype=bf16, device=dev)
            self.expert_scale = None
            self.expert_y = self.expert_x   # the identity expert by aliasing
        self.csend = torch.empty((n, self.RB, H), dtype=bf16, device=dev)
        self.crecv = torch.empty((n, T * R, H), dtype=bf16, device=dev)
        self.out = torch.empty((n, T, H), dtype=bf16, device=dev)
        self.plans = None

    # ------------------------------------------------------------------ steps
    def layout_step(self, stream=None):
        """moe_layout on every rank's ids (self.idx, filled by the routing exchange)."""
        check(lib().moe_layout(ctypes.byref(self.dims), self.idx.data_ptr(), ctypes.byref(self.layout),
                               _stream(stream)), "moe_layout")

    def layout_arrays(self) -> dict:
        """Device views of the layout's count and offset arrays."""
        base = self.workspace.data_ptr()
        N, E, L = self.N, self.E, self.L
        shapes = {"cnt": (N, E), "C": (N, N), "soff": (N, E), "roff": (N, N), "rtot": (N,), "ecnt": (N, L),
                  "eoff": (N, L, N), "pos": (N, self.T, self.R), "slot": (N, self.T, self.R)}
        out = {}
        for k, shp in shapes.items():
            off = getattr(self.layout, k) - base
            out[k] = self.workspace[off:off + 4 * int(np.prod(shp))].view(torch.int32).view(shp)
        return out

    def make_plans(self):
        """The four slice lists of this window (host; reads C, soff and roff back from the device;
        a single window exchanges nothing and reads nothing)."""
        if len(self.bounds) == 2:
            self.plans = {(direction, sending): [] for direction in (0, 1) for sending in (0, 1)}
            return self.plans
        a = self.layout_arrays()
        C, soff, roff = (a[k].cpu().numpy() for k in ("C", "soff", "roff"))
        self.plans = {(direction, sending): exchange_plan(self.dims, C, soff, roff, self.bounds, self.me, direction,
                                                          sending)
                      for direction in (0, 1) for sending in (0, 1)}
        return self.plans

    def dispatch_send(self, x_local: torch.Tensor, stream=None):
        """x_local [n, T, H] bf16: the window's tokens packed (quantised inside the pack for fp8)
        and the slices inside the window written."""
        fn = lib().moe_quantize_dispatch_send if self.fp8 else lib().moe_dispatch_send
        check(fn(ctypes.byref(self.dims), ctypes.byref(self.layout), x_local.data_ptr(), self.send.data_ptr(),
                 self.recv.data_ptr(), _stream(stream)), "dispatch send (window)")

    def dispatch_recv(self, stream=None):
        check(lib().moe_dispatch_recv(ctypes.byref(self.dims), ctypes.byref(self.layout), self.recv.data_ptr(),
                                      self.expert_x.data_ptr(),
                                      None if self.expert_scale is None else self.expert_scale.data_ptr(),
                                      _stream(stream)), "moe_dispatch_recv (window)")

    def expert_identity(self, stream=None):
        check(lib().moe_expert_identity(ctypes.byref(self.dims), ctypes.byref(self.layout), self.expert_x.data_ptr(),
                                        None if self.expert_scale is None else self.expert_scale.data_ptr(),
                                        self.expert_y.data_ptr(), _stream(stream)), "moe_expert_identity (window)")

    def combine_send(self, stream=None):
        check(lib().moe_combine_send(ctypes.byref(self.dims), ctypes.byref(self.layout), self.expert_y.data_ptr(),
                                     self.csend.data_ptr(), self.crecv.data_ptr(), _stream(stream)),
              "moe_combine_send (window)")

    def combine_recv(self, w_local: torch.Tensor, stream=None):
        check(lib().moe_combine_recv(ctypes.byref(self.dims), ctypes.byref(self.layout), self.crecv.data_ptr(),
                                     w_local.data_ptr(), self.out.data_ptr(), _stream(stream)),
              "moe_combine_recv (window)")

    def status(self, stream=None) -> tuple[int, int]:
        bits = ctypes.c_uint32(0)
        code = lib().moe_status_sync(ctypes.byref(self.layout), _stream(stream), ctypes.byref(bits))
        return int(code), int(bits.value)

    # ------------------------------------------------------------------ slice views
    def slice_views(self, direction: int, sending: int) -> list[tuple[int, int, int, torch.Tensor]]:
        """(peer, s, d, rows view) of each slice of the plan: send / receive rows for
        dispatch, combine-send / combine-receive rows for combine."""
        if direction == 0:
            buf = (self.send if sending else self.recv).view(-1, self.B)
        else:
            buf = (self.csend if sending else self.crecv).view(-1, self.H)
        return [(peer, s, d, buf[r0:r0 + rows]) for peer, s, d, rows, r0 in self.plans[(direction, sending)]]


class DistTransport:
    """Slices between processes of a torch.distributed group: window g is group rank g."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group

    def gather_routing(self, shard: ShardedEP, idx_local: torch.Tensor):
        """All windows' expert ids into shard.idx (windows of equal size)."""
        d = self.dist
        if d.get_world_size(self.group) == 1:
            shard.idx.copy_(idx_local)
            return
        d.all_gather_into_tensor(shard.idx, idx_local.contiguous(), group=self.group)

    def exchange(self, shards: list[ShardedEP], direction: int):
        """Sends every remote slice of this process's window and receives every one for it."""
        for shard in shards:
            self.exchange_views([(p, v) for p, _, _, v in shard.slice_views(direction, 1)],
                                [(p, v) for p, _, _, v in shard.slice_views(direction, 0)])

    def exchange_views(self, sends, recvs):
        """One message per slice: sends [(peer window, rows)], recvs [(peer window, rows)], each
        list in the plan's (s, d) order, so that the k-th send of window p to window q meets
        the k-th receive of q from p."""
        d = self.dist
        ops = [d.P2POp(d.isend, v, self._global(peer), group=self.group) for peer, v in sends]
        ops += [d.P2POp(d.irecv, v, self._global(peer), group=self.group) for peer, v in recvs]
        if ops:
            for w in d.batch_isend_irecv(ops):
                w.wait()

    def _global(self, peer: int) -> int:
        return peer if self.group is None else self.dist.get_global_rank(self.group, peer)


class LocalTransport:
    """Slices between windows held by one process (all on one device): a copy per slice."""

    def gather_routing(self, shards: list[ShardedEP], idx_parts: list[torch.Tensor]):
        full = torch.cat([p.reshape(-1, *p.shape[1:]) for p in idx_parts], dim=0)
        for sh in shards:
            sh.idx.copy_(full)

    def exchange(self, shards: list[ShardedEP], direction: int):
        recvs = {}
        for q, sh in enumerate(shards):
            for peer, s, d, v in sh.slice_views(direction, 0):
                recvs[(peer, q, s, d)] = v
        for p, sh in enumerate(shards):
            for peer, s, d, v in sh.slice_views(direction, 1):
                recvs.pop((p, peer, s, d)).copy_(v)
        assert not recvs, "every planned receive has its send"


def sharded_forward(shards: list[ShardedEP], transport, x_parts, idx_parts, w_parts, plan: bool = True):
    """One whole pass of the windows this process holds (one with DistTransport, all of them
    with LocalTransport), phase by phase. x_parts / idx_parts / w_parts: each window's tokens
    [n, T, H] bf16, ids [n, T, R] int32 and weights [n, T, R] fp32, on the device. With
    plan=False the slice lists of the previous pass are reused (same routing)."""
    if isinstance(transport, LocalTransport):
        transport.gather_routing(shards, idx_parts)
    else:
        for sh, idx in zip(shards, idx_parts):
            transport.gather_routing(sh, idx)
    for sh in shards:
        sh.layout_step()
    if plan or any(sh.plans is None for sh in shards):
        for sh in shards:
            sh.make_plans()
    for sh, x in zip(shards, x_parts):
        sh.dispatch_send(x)
    transport.exchange(shards, 0)
    for sh in shards:
        sh.dispatch_recv()
        sh.expert_identity()
        sh.combine_send()
    transport.exchange(shards, 1)
    for sh, w in zip(shards, w_parts):
        sh.combine_recv(w)
    return [sh.out for sh in shards]
