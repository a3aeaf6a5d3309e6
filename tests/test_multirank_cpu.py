"""The N > 1 bench path on the CPU: two gloo ranks.

The loss shards by tokens with no data-path collective: each rank runs its
own batch, and only the timing is combined (max over ranks, whole-job value
= every rank's tokens over the slowest rank's time).  These tests run that
host logic with world_size 2 over gloo on 127.0.0.1, and check that the
token-sharded means recombine into the single-batch mean the oracle gives.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist

    import bench
    import lossk_inputs as li
    import oracle
    r, w, loc = bench.dist_init()
    assert (r, w, loc) == (rank, world, rank)
    bench.barrier(w)
    ms = 10.0 + 5.0 * rank                          # rank 1 is the slow one
    mx = bench.max_over_ranks(ms, w)
    val = bench.aggregate(2048, w, mx)
    # each rank draws its own batch of the same model and computes its shard's sums
    x = li.make("tiny_fp32_ce", seed=0, batch=rank)
    f = oracle.ce_fwd(x["hidden"], x["weight"], x["targets"], chunk=16)
    q.put((rank, mx, val, f["total"] * len(x["targets"]), len(x["targets"])))
    dist.destroy_process_group()


def test_two_gloo_ranks_timing_and_sharding():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, val, _, _ in res:
        assert mx == 15.0
        assert val == pytest.approx(2 * 2048 / 0.015)
    # token sharding: the sum of the shards' loss sums over all tokens equals the
    # mean of the concatenated batch
    import lossk_inputs as li
    import oracle
    xs = [li.make("tiny_fp32_ce", seed=0, batch=r) for r in range(world)]
    H = np.concatenate([x["hidden"] for x in xs])
    y = np.concatenate([x["targets"] for x in xs])
    Wt = xs[0]["weight"]
    assert all(np.array_equal(x["weight"], Wt) for x in xs)   # same weight on every rank
    whole = oracle.ce_fwd(H, Wt, y, chunk=16)["total"]
    assert sum(r[3] for r in res) / sum(r[4] for r in res) == pytest.approx(whole, rel=1e-13)


def test_reference_arm_runs_on_rank0_only(monkeypatch):
    import bench
    a = type("A", (), {"steps": 1, "warmup": 0})()
    assert bench.run_reference(a, 1, 2) is None
