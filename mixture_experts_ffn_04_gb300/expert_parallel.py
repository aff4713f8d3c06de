"""Expert-parallel exchange for the routed experts ("Fused MoE Kernel Notes"
describes the non-EP fused path; this is its expert-parallel form).

Every rank keeps its own tokens (data parallel): it routes and permutes them
locally, so its grouped rows x_perm are expert-major with offsets[E + 1].  The
E experts are split into contiguous ranges, one per rank.  Two exchanges move
rows between ranks, and nothing else changes:

  dispatch  for every owner p and every expert e that p owns, the rows of e
            in this rank's x_perm (one contiguous slice, offsets[e] ..
            offsets[e + 1]) go to p, which receives the slices of all source
            ranks straight into an expert-major buffer: expert e's rows from
            rank 0, then from rank 1, ...  The owner then runs the grouped
            gate/up and down GEMMs over its E_local experts with the local
            offsets, exactly as the single-GPU layer does over E.
  return    the owner's output rows go back the same way: the slice of
            (source r, expert e) lands at offsets_r[e] of rank r's y_perm,
            which then feeds the local combine (gather with scatter_index and
            the routing weights).

The plan needs every rank's per-expert counts: one all_gather of E int32 per
rank.  The row exchanges are batched point-to-point messages, one per (peer,
owned expert) with rows, so no reorder step is needed on either side.  Works
with any torch.distributed backend that has isend/irecv (NCCL on GPUs; gloo on
CPU); with world size 1 both exchanges are copies.
"""
from __future__ import annotations

from typing import List, Optional, Tuple

import torch


def expert_ranges(num_experts: int, world: int) -> List[Tuple[int, int]]:
    """Contiguous expert ranges [e0, e1) per rank, sizes differing by at most 1."""
    base, extra = divmod(num_experts, world)
    out, e = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((e, e + n))
        e += n
    return out


class ExpertParallel:
    """Expert-parallel plan and exchanges for one layer call.

    counts: this rank's per-expert row counts [E] (int32, any device).  After
    plan(): local_counts [E_local] (rows this rank computes per owned expert)
    and local_offsets [E_local + 1]."""

    def __init__(self, num_experts: int, group=None):
        import torch.distributed as dist
        self.dist = dist if (dist.is_available() and dist.is_initialized()) else None
        self.group = group
        self.world = self.dist.get_world_size(group) if self.dist else 1
        self.rank = self.dist.get_rank(group) if self.dist else 0
        self.E = num_experts
        self.ranges = expert_ranges(num_experts, self.world)
        self.e0, self.e1 = self.ranges[self.rank]
        self.all_counts = None

    # -- plan ---------------------------------------------------------------
    def plan(self, counts: torch.Tensor):
        """Gather every rank's per-expert counts; returns (local_counts,
        local_offsets) of the experts this rank owns."""
        c = counts.to(torch.int64).reshape(1, self.E)
        if self.world > 1:
            bufs = [torch.empty_like(c) for _ in range(self.world)]
            self.dist.all_gather(bufs, c.contiguous(), group=self.group)
            allc = torch.cat(bufs, 0)
        else:
            allc = c.clone()
        self.all_counts = allc.cpu()                      # [world, E]
        local = self.all_counts[:, self.e0:self.e1]       # [world, E_local]
        self.local_counts = local.sum(0)                  # [E_local]
        self.local_offsets = torch.zeros(self.e1 - self.e0 + 1, dtype=torch.int64)
        self.local_offsets[1:] = torch.cumsum(self.local_counts, 0)
        # where (source r, expert e) starts in the owner's expert-major buffer
        self.recv_start = torch.zeros_like(local)
        for j in range(self.e1 - self.e0):
            col = local[:, j]
            self.recv_start[:, j] = self.local_offsets[j] + torch.cumsum(col, 0) - col
        return self.local_counts.to(torch.int32), self.local_offsets.to(torch.int32)

    def _my_offsets(self):
        c = self.all_counts[self.rank]
        off = torch.zeros(self.E + 1, dtype=torch.int64)
        off[1:] = torch.cumsum(c, 0)
        return off

    # -- exchanges ----------------------------------------------------------
    def _exchange(self, send_rows, recv_rows, sends, recvs):
        """sends / recvs: lists of (peer, start, count) row slices of
        send_rows / recv_rows."""
        local = [(s, r) for s, r in zip(
            [x for x in sends if x[0] == self.rank], [x for x in recvs if x[0] == self.rank])]
        for (_, s0, n), (_, r0, m) in local:
            assert n == m
            recv_rows[r0:r0 + n].copy_(send_rows[s0:s0 + n])
        ops = []
        if self.world > 1:
            P2POp, isend, irecv = self.dist.P2POp, self.dist.isend, self.dist.irecv
            for peer, s0, n in sends:
                if peer != self.rank and n > 0:
                    ops.append(P2POp(isend, send_rows[s0:s0 + n].contiguous(), peer, self.group))
            pending = []
            for peer, r0, n in recvs:
                if peer != self.rank and n > 0:
                    buf = torch.empty((n,) + tuple(recv_rows.shape[1:]), dtype=recv_rows.dtype,
                                      device=recv_rows.device)
                    ops.append(P2POp(irecv, buf, peer, self.group))
                    pending.append((r0, n, buf))
            if ops:
                for req in self.dist.batch_isend_irecv(ops):
                    req.wait()
            for r0, n, buf in pending:
                recv_rows[r0:r0 + n].copy_(buf)

    def dispatch(self, x_perm: torch.Tensor) -> torch.Tensor:
        """This rank's grouped rows [T*k, H] -> the rows of its owned experts
        from every rank, expert-major [local_offsets[-1], H]."""
        off = self._my_offsets()
        out = torch.empty((int(self.local_offsets[-1]),) + tuple(x_perm.shape[1:]),
                          dtype=x_perm.dtype, device=x_perm.device)
        sends, recvs = [], []
        for p, (e0, e1) in enumerate(self.ranges):
            for e in range(e0, e1):
                sends.append((p, int(off[e]), int(self.all_counts[self.rank, e])))
        for src in range(self.world):
            for j, e in enumerate(range(self.e0, self.e1)):
                recvs.append((src, int(self.recv_start[src, j]), int(self.all_counts[src, e])))
        self._exchange(x_perm, out, self._order(sends), self._order(recvs))
        return out

    def combine_back(self, y_local: torch.Tensor, y_perm: torch.Tensor) -> torch.Tensor:
        """The owner's output rows [local_offsets[-1], H] back to their source
        ranks: fills this rank's y_perm [T*k, H] (expert-major, its own
        offsets) and returns it."""
        off = self._my_offsets()
        sends, recvs = [], []
        for src in range(self.world):
            for j, e in enumerate(range(self.e0, self.e1)):
                sends.append((src, int(self.recv_start[src, j]), int(self.all_counts[src, e])))
        for p, (e0, e1) in enumerate(self.ranges):
            for e in range(e0, e1):
                recvs.append((p, int(off[e]), int(self.all_counts[self.rank, e])))
        self._exchange(y_local, y_perm, self._order(sends), self._order(recvs))
        return y_perm

    @staticmethod
    def _order(msgs):
        # one fixed order on both sides of every peer pair: by peer, then slice
        return sorted(msgs, key=lambda m: (m[0], m[1]))


def ep_layer_forward(m, layer, x: torch.Tensor, ep: Optional[ExpertParallel] = None,
                     stream=None) -> torch.Tensor:
    """The routed-expert layer with its experts split over the ranks of
    `ep` (CUDA, through the library's entry points): route and permute the
    local tokens, dispatch, grouped gate/up and down over the owned experts,
    return, combine.  Layers with a shared MLP, an input RMSNorm or MXFP8
    weights are not covered (the shared MLP is data parallel and can be added
    to the combine by the caller)."""
    wl, s, ws = layer.wl, layer.shape, layer.ws
    if wl.I_sh or getattr(wl, "input_norm", False) or getattr(wl, "weights", "act") != "act":
        raise ValueError("ep_layer_forward covers the routed experts only")
    ep = ep or ExpertParallel(wl.E)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    dev, dt = x.device, x.dtype
    i32 = dict(dtype=torch.int32, device=dev)
    idx, tw = torch.empty(T, k, **i32), torch.empty(T, k, dtype=torch.float32, device=dev)
    m.moe_route(s, x, layer.inputs["w_router"], idx, tw, None, ws, stream)
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    sidx, row_token = torch.empty(T, k, **i32), torch.empty(T * k, **i32)
    x_perm = torch.empty(T * k, H, dtype=dt, device=dev)
    m.moe_permute(s, x, idx, counts, offsets, sidx, row_token, x_perm, ws, stream)
    _, loff = ep.plan(counts)   # reads the counts back: waits for the permute
    x_loc = ep.dispatch(x_perm)
    R = x_loc.shape[0]
    E_loc = ep.e1 - ep.e0
    y_loc = torch.empty(R, H, dtype=dt, device=dev)
    if R > 0 and E_loc > 0:
        h = torch.empty(R, I, dtype=dt, device=dev)
        off_dev = loff.to(device=dev)
        gw, uw, dw = layer.inputs["w_gate"], layer.inputs["w_up"], layer.inputs["w_down"]
        m.moe_grouped_swiglu(s, x_loc, gw[ep.e0:ep.e1], uw[ep.e0:ep.e1], I * H, off_dev, E_loc,
                             R, I, h, ws, stream)
        m.moe_grouped_down(s, h, dw[ep.e0:ep.e1], H * I, off_dev, E_loc, R, I, y_loc, ws, stream)
    y_perm = torch.empty(T * k, H, dtype=dt, device=dev)
    ep.combine_back(y_loc, y_perm)
    y = torch.empty_like(x)
    m.moe_combine(s, y_perm, sidx, tw, None, None, y, stream)
    return y
