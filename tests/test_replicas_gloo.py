"""The bench's multi-process path on CPU: two gloo ranks run the same
rank-side helpers bench.py uses under torchrun (independent replicas, the
max-over-ranks time, the whole-job rate) and must agree on the job's
numbers."""
import json
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        layer_seeds, token_seed = bench.replica_seeds(rank, 4)
        dist.barrier()
        # each rank timed its own K steps; the job ends with the slowest one
        own_ms = 10.0 + 2.5 * rank
        ms = bench.max_over_ranks(dist, own_ms, "cpu")
        rate = bench.job_rate(200 * 8, world, ms)
        with open(os.path.join(out_dir, "rank%d.txt" % rank), "w") as f:
            json.dump([ms, rate, layer_seeds, token_seed], f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_job_numbers(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    rows = []
    for rank in range(world):
        ms, rate, layer_seeds, token_seed = json.load(open(tmp_path / ("rank%d.txt" % rank)))
        rows.append((ms, rate, layer_seeds, token_seed))
    # both ranks report the slowest rank's time and the same whole-job rate
    assert rows[0][0] == rows[1][0] == 12.5
    assert rows[0][1] == rows[1][1] == pytest.approx(200 * 8 * 2 / 12.5e-3)
    # replicas: disjoint layer seeds and different token streams
    assert not set(rows[0][2]) & set(rows[1][2])
    assert rows[0][3] != rows[1][3]


def test_single_process_helpers():
    import bench
    assert bench.max_over_ranks(None, 3.25, "cpu") == 3.25
    assert bench.job_rate(1000, 1, 500.0) == pytest.approx(2000.0)
    seeds, tok = bench.replica_seeds(0, 3)
    assert seeds == [0, 1, 2] and tok == 0
