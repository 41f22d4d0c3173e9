"""The benchmark's multi-rank host logic on CPU ranks (gloo, world size 2).

Each rank runs its own replica of the workload; the only cross-rank operations are
the barrier and the max over ranks of the step time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, lr = bench.dist_env()
    assert (w, r, lr) == (world, rank, rank)
    bench.barrier(world)
    step_ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
    results[rank] = bench.reduce_max(step_ms, world, "cpu")
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(results) == {0: 15.0, 1: 15.0}


def test_reference_arm_only_prints_on_rank_zero(monkeypatch):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup, reference_seconds = 1, 0, 1.0

    assert bench.run_reference(A()) is None


def test_valid_pair_count_matches_oracle_routes():
    import numpy as np

    import bench
    import irs_synth
    from oracle import irs_oracle as O

    wl = irs_synth.custom(300, 2, 1, 64, 128, Hi=2, Di=64, c=4, budget=32, doc_lens=[120, 3, 177], seed=2)
    r = O.index_routes(wl.arrays["qI"], wl.arrays["kI"], wl.arrays["w"], wl.cu_seqlens, wl.c, wl.budget)
    np.testing.assert_array_equal(bench.valid_per_row(wl), (r >= 0).sum(axis=1))
