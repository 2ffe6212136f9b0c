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


def _failing_worker(rank, world, port, mode, q):
    """Rank 1 fails between steps (it raises before the barrier, or stalls past the
    timeout without joining it); rank 0 must see an error from its next collective
    within the bench's bounded process-group timeout, not hang."""
    import time

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    os.environ["RANK"] = str(rank)
    os.environ["WORLD_SIZE"] = str(world)
    import bench
    bench.init_dist("gloo", timeout_s=5.0)
    if rank == 1:
        if mode == "stall":
            time.sleep(20.0)
            os._exit(0)
        os._exit(3)                 # the rank dies without joining
    t0 = time.perf_counter()
    try:
        bench.barrier(True)
        bench.max_over_ranks(1.0, True, torch.device("cpu"))
        q.put((rank, "completed", time.perf_counter() - t0))
    except Exception as e:      # the collective's error is the detection
        q.put((rank, type(e).__name__, time.perf_counter() - t0))
    q.close()
    q.join_thread()             # the result is in the pipe before the process leaves
    os._exit(0)


@pytest.mark.parametrize("mode", ["dies", "stall"])
def test_a_failed_rank_ends_the_others_collectives(mode):
    ctx = mpl.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_failing_worker, args=(r, 2, port, mode, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        rank, outcome, dt = q.get(timeout=60)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert rank == 0
    assert outcome != "completed"
    assert dt < 15.0                # the 5 s timeout, not the stalled rank's 20 s
