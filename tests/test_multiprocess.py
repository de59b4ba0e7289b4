"""The N > 1 benchmark path on CPU: two gloo ranks aggregate like the GPU run.

Decode requests are independent, so ranks share nothing but the timing
reductions: whole-job throughput is every rank's bytes over the slowest
rank's time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ranks = bench.Ranks(backend="gloo")
    try:
        ranks.barrier()
        # rank r processed (r + 1) GB in (r + 1) seconds over 10 steps
        agg = bench.aggregate(ranks, per_rank_bytes=(rank + 1) * 1e8,
                              elapsed_s=float(rank + 1), steps=10)
        results[rank] = (ranks.world, ranks.rank, agg["value_gbs"],
                         agg["ms_per_step"], agg["slowest_s"])
    finally:
        ranks.close()


def test_two_gloo_ranks_aggregate_bytes_over_slowest_time():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as manager:
        results = manager.dict()
        mp.start_processes(_worker, args=(world, port, results), nprocs=world,
                           join=True, start_method="spawn")
        res = dict(results)
    assert sorted(res) == [0, 1]
    for rank, (w, r, value, ms, slowest) in res.items():
        assert w == 2 and r == rank
        # (1e8 + 2e8) bytes x 10 steps over the slowest rank's 2 s
        assert value == pytest.approx(3e8 * 10 / 2.0 / 1e9)
        assert ms == pytest.approx(2.0 * 1e3 / 10)
        assert slowest == 2.0


def test_single_process_needs_no_process_group():
    import bench
    ranks = bench.Ranks()
    assert ranks.world == 1 and ranks.dist is None
    agg = bench.aggregate(ranks, per_rank_bytes=5e8, elapsed_s=0.5, steps=5)
    assert agg["value_gbs"] == pytest.approx(5e8 * 5 / 0.5 / 1e9)
