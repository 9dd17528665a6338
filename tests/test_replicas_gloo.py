"""The multi-GPU path is replicas only: bench.py's aggregation (max time over
ranks, layers summed over ranks) checked with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    per_rank_seconds = 0.010 * (rank + 1)          # rank 1 is the slow one
    agg = bench.aggregate(per_rank_seconds, layers_per_rank=400, world=world)
    q.put((rank, agg))
    dist.destroy_process_group()


def test_replica_aggregation_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        agg = out[r]
        assert agg["seconds"] == pytest.approx(0.020)      # the slowest rank's time
        assert agg["total_layers"] == 800                  # every rank's layers
        assert agg["us_per_layer"] == pytest.approx(0.020 * 1e6 / 800)


def test_single_process_is_identity():
    import bench
    agg = bench.aggregate(0.5, layers_per_rank=1000, world=1)
    assert agg["seconds"] == 0.5 and agg["total_layers"] == 1000
