"""The multi-rank host logic of bench.py on CPU: two gloo ranks over 127.0.0.1.

The decode path shards by sequence with no exchange; the only cross-rank steps are
the barrier around the timed region, the max over ranks of the elapsed time and the
sum over ranks of the processed tokens (the whole-job value).  Each rank also draws
its own sequences (seed offset by rank).
"""
import multiprocessing as mpl
import os
import socket

import pytest
import torch


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    import bench
    from looped_transformer_cross_gb300.synth import WORKLOADS, make_decode_inputs
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dev = torch.device("cpu")
        bench.barrier(True)
        mx = bench.max_over_ranks(1.5 * (rank + 1), True, dev)
        sm = bench.sum_over_ranks(10.0 * (rank + 1), True, dev)
        w = WORKLOADS["tiny_f32"]
        inp = make_decode_inputs(w, 20260000 + 1 + 1000 * rank)
        q.put((rank, mx, sm, float(inp["cache_k"].sum())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_tokens():
    ctx = mpl.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    try:
        for _ in range(2):
            rank, mx, sm, ck = q.get(timeout=120)
            res[rank] = (mx, sm, ck)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    assert res[0][0] == res[1][0] == pytest.approx(3.0)      # max of 1.5, 3.0
    assert res[0][1] == res[1][1] == pytest.approx(30.0)     # 10 + 20
    assert res[0][2] != res[1][2]                            # each rank holds its own sequences
