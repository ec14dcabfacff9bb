"""World-size-2 gloo tests (CPU) of the benchmark's multi-rank host logic:
each rank draws its own shard of independent sequences, and the only
collective is the max over ranks of the timings (no data-path exchange)."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from transformer_scaled_dot_fwd_gb300 import workloads as wl

    w_env, r_env, _ = bench.dist_env()
    assert (w_env, r_env) == (world, rank)
    d = bench.init_dist(world, "gloo")
    try:
        bench.barrier(d)
        # the slowest rank's time is the job's time
        got = bench.max_over_ranks(d, 1.0 + rank * 2.5, torch.device("cpu"))
        # each rank's shard: the same workload shape, its own seed
        small = wl.PrefillWorkload("shard", 1, 2, 8, 64, "bf16", True, seed=wl.PREFILL.seed)
        q, _, _, _ = wl.prefill_inputs(small, device="cpu", seed=small.seed + 1000 * rank)
        gathered = [torch.zeros_like(q, dtype=torch.float32) for _ in range(world)]
        dist.all_gather(gathered, q.float())  # test-only: compare shards across ranks
        cfg = bench.config_dict(wl.PREFILL, world)
        results[rank] = (got, bool(torch.equal(gathered[0], gathered[1])), cfg["global_batch"])
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(2, port, results), nprocs=2, join=True)
        res = dict(results)
    assert res[0][0] == pytest.approx(3.5) and res[1][0] == pytest.approx(3.5)
    assert res[0][1] is False, "both ranks drew the same shard"
    assert res[0][2] == 2 * 4 and res[1][2] == 8


def test_single_process_needs_no_process_group():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 2.0, torch.device("cpu")) == 2.0
