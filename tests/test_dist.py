"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): each rank verifies its own
distinct requests, and the step time / position counts reduce across ranks."""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, wsz, _ = bench.dist_env()
    assert (r, wsz) == (rank, world)
    reqs = bench.shard_requests(4, rank)
    w = W.get("c2", B=4, V=2000, tau=0.5)
    d = W.generate(w, requests=reqs)
    mx = bench.max_over_ranks(1.0 + rank, world)
    tot = bench.sum_over_ranks(float(d["k_per_row"].sum()), world)
    bench.barrier(world)
    out[rank] = (list(reqs), mx, tot, float(d["p"][0, 0, :8].astype(np.float64).sum()))
    dist.destroy_process_group()


def test_two_ranks_shard_and_reduce():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of a process that runs threads
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    (r0, mx0, t0, s0), (r1, mx1, t1, s1) = res[0], res[1]
    assert set(r0).isdisjoint(r1) and len(r0) == len(r1) == 4
    assert mx0 == mx1 == 2.0  # max over ranks
    assert t0 == t1 == 2 * 4 * 5  # sum over ranks of sum_b K_b
    assert s0 != s1  # distinct requests, distinct logits
