"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): each rank gets its own
batch, the step time is the max over ranks and the throughput counts every rank's nodes."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench
from speculative_decoding_tree_mask_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, wsz, local = bench.dist_env()
    bench.init_dist(wsz, "gloo")
    w = W.WORKLOADS["large_tree"].scaled(B=3, N=8, V=64)
    x = W.make(w, seed=bench.rank_seed(w, r))
    my_ms = 1.0 + r                                   # rank 1 is the slow one
    ms = bench.max_over_ranks(my_ms, wsz, "cpu")
    bench.barrier(wsz)
    value = bench.aggregate_throughput(wsz, w.draft_nodes, ms)
    q.put((r, ms, value, x["parent_np"].tolist(), x["logits"][0, 0, :4].tolist()))
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ms0, v0, par0, lg0), (r1, ms1, v1, par1, lg1) = out
    assert ms0 == ms1 == 2.0                          # max over ranks
    assert v0 == v1 == pytest.approx(2 * 3 * 7 / 2e-3)
    assert lg0 != lg1                                 # independent batches per rank


def test_single_rank_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
