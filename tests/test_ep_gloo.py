"""Expert-parallel layer on CPU: two (or three) gloo ranks run the
orchestration of quantized_expert_ffn_warp_gb300.ep (route, dispatch by
destination rank, all-to-all of rows and local expert ids, the owned
experts, all-to-all back, combine) with a CPU backend built on the oracle.
Each rank's outputs must equal, bit for bit, the single-process oracle
forward of the same tokens: the bookkeeping of the exchange (who owns which
expert, in which order rows go and come back) loses nothing.  The GPU side
of the same steps (the dispatch and combine kernels) is checked against the
same reference in tests/test_gpu_ep.py."""
import json
import math
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from quantized_expert_ffn_warp_gb300 import ep, synth  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def dispatch_reference(idx, n_experts, world):
    """Send positions grouped by destination rank, pair order kept inside a
    rank; local expert ids; rows per destination."""
    flat = np.asarray(idx).reshape(-1)
    dest = np.array([ep.owner(int(e), n_experts, world) for e in flat])
    order = np.argsort(dest, kind="stable")
    pos = np.empty(len(flat), np.int64)
    pos[order] = np.arange(len(flat))
    local = np.array([int(e) - ep.first_expert(int(d), n_experts, world)
                      for e, d in zip(flat, dest)])
    counts = [int((dest == r).sum()) for r in range(world)]
    return pos, local[order], counts


class OracleBackend:
    """The compute steps on the CPU in fp64 with the oracle: the exchange
    carries fp64 rows, so the result can be compared bit for bit."""

    def __init__(self, packed, rank, world):
        import oracle
        self.o = oracle
        self.packed = packed
        self.spec = packed.spec
        self.lo = ep.first_expert(rank, self.spec.n_experts, world)

    def route(self, x16):
        lg = self.o.router_logits(x16, self.packed.router_w, self.packed.router_bias)
        r = self.o.topk(lg, self.spec.top_k)
        return r[0], r[2]            # idx int32, fp64 weights

    def dispatch(self, x16, idx, n_experts, world):
        pos, local, counts = dispatch_reference(idx, n_experts, world)
        k = self.spec.top_k
        rows = np.empty((len(pos), x16.shape[1]), np.int16)
        rows[pos] = x16.view(np.int16)[np.arange(len(pos)) // k]
        send_e = np.empty(len(pos), np.int32)
        send_e[:] = local
        # fp16 rows on the wire (gloo has no int16 all-to-all)
        return (torch.from_numpy(rows.view(np.float16)), torch.from_numpy(send_e), pos, counts)

    def experts(self, rows, local_ids):
        rows = rows.numpy().view(np.uint16)
        ids = local_ids.numpy()
        y = np.zeros((len(ids), self.spec.hidden), np.float64)
        for e in np.unique(ids):
            sel = np.nonzero(ids == e)[0]
            y[sel] = self.o.expert_ffn(self.packed, int(e) + self.lo, rows[sel])
        return torch.from_numpy(y)

    def shared(self, x16):
        if not self.spec.has_shared:
            return None
        return self.o.expert_ffn(self.packed, -1, x16)

    def combine(self, x16, w, pos, y_back, y_sh):
        """x + sum_j w_j y_j (slot order) + sigmoid(x . wg) y_sh, in fp64,
        rounded once to fp16: the oracle's own combine order."""
        xf = x16.view(np.float16).astype(np.float64)
        y = y_back.numpy()
        n, k = w.shape
        out = xf.copy()
        for j in range(k):
            out += w[:, j:j + 1] * y[pos.reshape(n, k)[:, j]]
        if y_sh is not None:
            g = self.packed.sh_gate_w.view(np.float16).astype(np.float64)
            # the gate as the oracle takes it: a sequential fp64 dot product
            # and the C library's exp
            gate = np.array([1.0 / (1.0 + math.exp(-sum(float(a) * float(b)
                                                        for a, b in zip(row, g))))
                             for row in xf])
            out += gate[:, None] * y_sh
        return out.astype(np.float16).view(np.uint16)


CASES = {
    # ragged shapes, 12 experts top-3 with a shared expert, split 6/6
    "ragged": (synth.LayerSpec("ragged_ep", hidden=384, inter=256, n_experts=12, top_k=3,
                               has_shared=True, shared_inter=256, zipf_s=0.8), 2),
    # 5 experts over 2 ranks (2 / 3): an uneven partition
    "uneven": (synth.LayerSpec("uneven_ep", hidden=256, inter=256, n_experts=5, top_k=2), 2),
    # 8 experts over 3 ranks
    "three": (synth.LayerSpec("three_ep", hidden=256, inter=384, n_experts=8, top_k=2,
                              zipf_s=1.0), 3),
}


def _rank_main(rank, world, port, out_dir, case, tie):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        spec, _ = CASES[case]
        packed = synth.make_layer(spec, seed=2)
        if tie:   # a zero router: every token picks experts 0..k-1, all on rank 0
            packed.router_w[:] = 0
            packed.router_bias = None
        n_per = 5 + rank            # ranks with different token counts
        x = synth.make_tokens(spec, n_per, seed=3, batch=rank)
        layer = ep.ExpertParallelLayer(OracleBackend(packed, rank, world), spec.n_experts, world,
                                       rank, pg=dist)
        out = layer.forward(x)
        ref = oracle.forward(packed, x)["out16"]
        with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
            json.dump({"equal": bool(np.array_equal(out, ref)),
                       "max_diff": float(np.abs(out.view(np.float16).astype(np.float64)
                                                - ref.view(np.float16).astype(np.float64)).max())},
                      f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case,tie", [("ragged", False), ("uneven", False), ("three", False),
                                      ("ragged", True)])
def test_expert_parallel_matches_single_process(tmp_path, case, tie):
    world = CASES[case][1]
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path), case, tie),
                       nprocs=world, join=True, start_method="spawn")
    for rank in range(world):
        r = json.load(open(tmp_path / ("rank%d.json" % rank)))
        assert r["equal"], (rank, r)


def test_partition_covers_every_expert_once():
    for E in (1, 5, 8, 12, 64, 512):
        for world in range(1, min(E, 8) + 1):
            owners = [ep.owner(e, E, world) for e in range(E)]
            assert owners == sorted(owners)
            for r in range(world):
                lo, hi = ep.first_expert(r, E, world), ep.first_expert(r + 1, E, world)
                assert owners[lo:hi] == [r] * (hi - lo)
            assert ep.first_expert(world, E, world) == E
