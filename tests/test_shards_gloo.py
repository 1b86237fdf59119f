"""Multi-rank host logic of bench.py on CPU with gloo, world size 2: process-group
set-up, barrier, max-over-ranks timing, distinct per-rank units, and the
whole-job aggregate. No data-path collective exists to test."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    from causal_head_attention_gb300.inputs import HEADLINE

    w_, r_, _ = bench.dist_setup()
    bench.barrier(w_)
    t = bench.max_over_ranks(10.0 + rank, w_)  # the slowest rank's time wins
    wl = bench.rank_workload(HEADLINE, r_)
    out.put((r_, w_, t, wl.seed, wl.B, wl.T))
    dist.destroy_process_group()


def test_two_rank_gloo_bench_logic():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 for r in res)
    assert all(r[2] == 11.0 for r in res)
    assert res[0][3] != res[1][3]  # distinct units per rank
    assert res[0][4:] == res[1][4:]  # same per-rank shape: weak scaling


def test_aggregate_counts_every_rank():
    import bench

    assert bench.aggregate_tflops(1e12, 1, 1000.0) == pytest.approx(1.0)
    assert bench.aggregate_tflops(1e12, 4, 2000.0) == pytest.approx(2.0)
