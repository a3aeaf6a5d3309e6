"""Vocabulary-parallel cross-entropy: the exchange between ranks, on the CPU.

Two gloo ranks (127.0.0.1) each hold one contiguous shard of the weight's
vocabulary rows.  Each computes its shard's partials and backward with the
oracle (the CPU stand-in for the shard kernels), and the exchange code of
output_projection_cross_gb300.vocab_parallel moves them: one all-gather of
the partials, one all-reduce of the d_hidden shares.  The combined loss, the
summed d_hidden and the concatenated d_weight shards must be the unsharded
oracle's.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _inputs():
    g = np.random.default_rng(90)
    n, d, V = 24, 16, 101
    H = g.standard_normal((n, d)).astype(np.float32)
    W = (g.standard_normal((V, d)) * 0.3).astype(np.float32)
    y = g.integers(0, V, n).astype(np.int64)
    y[:4] = [0, V - 1, 50, 51]               # both ends and both sides of the cut
    mask = np.ones(n, np.uint8)
    mask[[2, 9]] = 0
    return H, W, y, mask


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world)})
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle
    from output_projection_cross_gb300 import vocab_parallel as vp
    dist.init_process_group("gloo")
    H, W, y, mask = _inputs()
    V = W.shape[0]
    v0, rows = vp.shard_range(V, world, rank)
    Ws = W[v0:v0 + rows]
    p = torch.from_numpy(oracle.ce_shard_fwd(H, Ws, y, v0, V))
    pa = vp.gather_partials(p)
    assert tuple(pa.shape) == (world, 3, len(y))
    c = oracle.ce_shard_combine(pa.numpy(), mask=mask, z_weight=0.02)
    dh, dw = oracle.ce_shard_bwd(H, Ws, y, v0, V, c["lse"], mask=mask, z_weight=0.02, grad_scale=1.3)
    dh = vp.sum_d_hidden(torch.from_numpy(dh)).numpy()
    q.put((rank, v0, rows, c, dh, dw))
    dist.destroy_process_group()


def test_shard_range_tiles_the_vocabulary():
    from output_projection_cross_gb300 import vocab_parallel as vp
    for V, world in ((151936, 2), (101, 2), (101, 3), (8, 8), (1000, 7)):
        prev = 0
        for r in range(world):
            v0, rows = vp.shard_range(V, world, r)
            assert v0 == prev and rows in (V // world, V // world + 1)
            prev = v0 + rows
        assert prev == V
    with pytest.raises(ValueError):
        vp.shard_range(3, 4, 0)


def test_two_gloo_ranks_exchange_recombines_the_loss():
    from conftest import build_lib
    build_lib()
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in range(world)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import oracle
    H, W, y, mask = _inputs()
    f = oracle.ce_fwd(H, W, y, mask=mask, z_weight=0.02)
    dH, dW = oracle.ce_bwd(H, W, y, mask=mask, z_weight=0.02, grad_scale=1.3)
    for rank, v0, rows, c, dh, dw in res:
        # every rank holds the whole vocabulary's loss and the summed d_hidden
        assert np.allclose(c["lse"], f["lse"], rtol=1e-14, atol=0)
        assert np.allclose(c["ce"], f["ce"], rtol=1e-13, atol=1e-15)
        assert c["total"] == pytest.approx(f["total"], rel=1e-13)
        assert np.allclose(dh, dH, rtol=1e-12, atol=1e-16)
        assert np.allclose(dw, dW[v0:v0 + rows], rtol=1e-12, atol=1e-16)
    assert res[0][1] == 0 and res[0][1] + res[0][2] == res[1][1] and res[1][1] + res[1][2] == W.shape[0]
