"""Expert-parallel MoE layer across ranks (one GPU each): the routed experts
are partitioned by id ("Strata" article, section 5.2: with two cards the
expert cache is sharded per card), rank r owning experts
[r*E//world, (r+1)*E//world).

A forward on every rank: route the rank's tokens, pack one activation row per
(token, slot) pair grouped by destination rank, exchange rows and local
expert ids with an all-to-all, run the owned experts on the received rows,
send the result rows back with a second all-to-all, and combine them with
the weights, the residual and the shared expert (every rank keeps its own
copy of the shared expert).

This module only orders the steps and exchanges the buffers: every step of
the layer runs in the library's kernels (moe_route_topk_noalloc,
moe_ep_dispatch, moe_forward_routed, moe_ep_combine) through CudaBackend;
the collective is torch.distributed's all_to_all_single (NCCL between GPUs).
"""
from __future__ import annotations

import numpy as np


def owner(e: int, n_experts: int, world: int) -> int:
    """Rank that owns expert e."""
    return ((e + 1) * world - 1) // n_experts


def first_expert(r: int, n_experts: int, world: int) -> int:
    """First expert id of rank r."""
    return r * n_experts // world


def exchange(pg, send, send_counts, recv_counts):
    """All-to-all of the rows of `send` (first dimension) with per-rank
    counts; returns the received rows in rank order.  Without a process group
    (one rank) the rows are returned as they are."""
    import torch
    if pg is None:
        return send[: sum(send_counts)]
    out = torch.empty((sum(recv_counts),) + tuple(send.shape[1:]), dtype=send.dtype,
                      device=send.device)
    pg.all_to_all_single(out, send[: sum(send_counts)].contiguous(),
                         output_split_sizes=list(recv_counts), input_split_sizes=list(send_counts))
    return out


def exchange_counts(pg, counts, world):
    """Each rank's row count for every other rank."""
    import torch
    if pg is None:
        return list(counts)
    send = torch.tensor([int(c) for c in counts], dtype=torch.int64)
    recv = torch.empty(world, dtype=torch.int64)
    pg.all_to_all_single(recv, send)
    return [int(v) for v in recv]


class ExpertParallelLayer:
    """One rank's part of an expert-parallel layer.  `backend` provides the
    compute steps (CudaBackend on a GPU); `pg` is torch.distributed (or None
    for a single rank).  Counts travel on `count_pg` (a CPU-capable group,
    e.g. gloo) when given, else on `pg`."""

    def __init__(self, backend, n_experts, world, rank, pg=None, count_pg=None):
        self.backend = backend
        self.E = n_experts
        self.world = world
        self.rank = rank
        self.pg = pg
        self.count_pg = count_pg if count_pg is not None else pg

    def forward(self, x):
        b = self.backend
        idx, w = b.route(x)
        send_x, send_e, pos, dest_counts = b.dispatch(x, idx, self.E, self.world)
        recv_counts = exchange_counts(self.count_pg, dest_counts, self.world)
        recv_x = exchange(self.pg, send_x, dest_counts, recv_counts)
        recv_e = exchange(self.pg, send_e, dest_counts, recv_counts)
        y_recv = b.experts(recv_x, recv_e)
        y_back = exchange(self.pg, y_recv, recv_counts, dest_counts)
        y_sh = b.shared(x)
        return b.combine(x, w, pos, y_back, y_sh)


class CudaBackend:
    """The compute steps on one GPU through the library's C ABI: routing by
    moe_route_topk_noalloc against the full router, dispatch and combine by
    moe_ep_dispatch / moe_ep_combine, the owned experts by a layer of those
    experts only (top_k = 1, residual = 0, no shared expert) and the shared
    expert by a one-expert layer, both called with moe_forward_routed."""

    def __init__(self, packed, rank, world, max_rows, device="cuda"):
        import torch
        from . import moe, synth
        spec = packed.spec
        self.spec = spec
        self.moe = moe
        E = spec.n_experts
        lo, hi = first_expert(rank, E, world), first_expert(rank + 1, E, world)
        self.router_w = torch.from_numpy(packed.router_w.view(np.int16)).to(device)
        self.router_b = (torch.from_numpy(packed.router_bias).to(device)
                         if packed.router_bias is not None else None)
        local = synth.PackedLayer(
            spec.with_(name=spec.name + "_ep%d" % rank, n_experts=hi - lo, top_k=1,
                       has_shared=False, shared_inter=0, zipf_s=None),
            [c[lo:hi] for c in packed.codes], [s[lo:hi] for s in packed.scales],
            [z[lo:hi] for z in packed.zeros], packed.router_w[lo:hi], None)
        self.local = moe.MoeLayer(local.spec, moe.upload(local, device), max_tokens=max_rows,
                                  residual=0)
        self.shared_layer = None
        if spec.has_shared:
            sh = synth.PackedLayer(
                spec.with_(name=spec.name + "_sh", inter=spec.shared_inter, n_experts=1,
                           top_k=1, has_shared=False, shared_inter=0, zipf_s=None),
                packed.sh_codes, packed.sh_scales, packed.sh_zeros,
                np.zeros((1, spec.hidden), np.uint16), None)
            self.shared_layer = moe.MoeLayer(sh.spec, moe.upload(sh, device),
                                             max_tokens=max_rows, residual=0)
            self.gate_w = torch.from_numpy(packed.sh_gate_w.view(np.int16)).to(device)
        self.ones = torch.ones(max_rows, dtype=torch.float32, device=device)
        self.zeros = torch.zeros(max_rows, dtype=torch.int32, device=device)

    def route(self, x):
        import torch
        n, H = x.shape
        E, k = self.spec.n_experts, self.spec.top_k
        chunk = max(1, self.moe.MOE_NOALLOC_MAX_SCORES // E)
        idx = torch.empty((n, k), dtype=torch.int32, device=x.device)
        w = torch.empty((n, k), dtype=torch.float32, device=x.device)
        for t0 in range(0, n, chunk):   # row slices of contiguous buffers stay contiguous
            self.moe.route_topk_noalloc(x[t0:t0 + chunk], self.router_w, self.router_b, k,
                                        idx=idx[t0:t0 + chunk], w=w[t0:t0 + chunk])
        return idx, w

    def dispatch(self, x, idx, n_experts, world):
        send_x, send_e, pos, counts, status = self.moe.ep_dispatch(x, idx, n_experts, world)
        return send_x, send_e, pos, counts.cpu().tolist()

    def experts(self, rows, local_ids):
        m = rows.shape[0]
        if m == 0:
            return rows
        return self.local.forward_routed(rows, local_ids.view(m, 1), self.ones[:m].view(m, 1))

    def shared(self, x):
        if self.shared_layer is None:
            return None
        n = x.shape[0]
        return self.shared_layer.forward_routed(x, self.zeros[:n].view(n, 1),
                                                self.ones[:n].view(n, 1))

    def combine(self, x, w, pos, y_back, y_sh):
        return self.moe.ep_combine(x, w, pos, y_back,
                                   self.gate_w if y_sh is not None else None, y_sh)

    def close(self):
        self.local.close()
        if self.shared_layer is not None:
            self.shared_layer.close()
