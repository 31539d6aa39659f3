"""The N > 1 benchmark path on CPU: two gloo ranks (127.0.0.1) run bench.py's aggregation, which
must take the slowest rank's time and count every rank's work (weak scaling, no data-path
collective).  Also checks that the per-rank workloads differ only by seed."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_total = [400.0, 1000.0][rank]  # rank 1 is the slow one
    work = 2.0e9                      # units per step on each rank
    ms_step, value = bench.aggregate(work, ms_total, 100, world)
    bench.barrier(world)
    q.put((rank, ms_step, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_slowest_time_and_sum_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms_step, value in res:
        assert ms_step == pytest.approx(10.0)              # max(400, 1000) / 100 steps
        assert value == pytest.approx(2 * 2.0e9 / 10e-3)    # both ranks' work / slowest time


def test_single_rank_aggregate_is_identity():
    import bench
    ms_step, value = bench.aggregate(5.0e8, 250.0, 50, 1)
    assert ms_step == pytest.approx(5.0) and value == pytest.approx(1e11)


def test_rank_seeds_give_same_shape_different_data():
    from paged_kv_cache_rope_gb300 import workloads as W
    for idx in (1, 4):
        a = W.workload(idx, seed=idx)
        b = W.workload(idx, seed=idx + 1000)  # what rank 1 of a torchrun job draws
        assert (a.new_len == b.new_len).all() and (a.past == b.past).all()
        assert a.pool.shape == b.pool.shape
        assert not torch.equal(a.q, b.q)
