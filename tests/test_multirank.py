"""The multi-rank host path of bench.py on CPU: two gloo ranks.

bench.py runs one replica per GPU (the path partitions by request, so there
is no data-path collective); what the ranks share is the barrier around the
timed region and the max over ranks of the measured time.  Both are checked
here with world size 2 on the gloo backend, plus the rule that only rank 0
runs and prints the reference arm.
"""
import contextlib
import io
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        bench.barrier(w)
        t = bench.max_over_ranks(10.0 + 5.0 * rank, w)   # rank 1 is the slow one
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            class A:
                steps, warmup = 1, 0
            if r != 0:
                bench.run_reference(A, r, w)            # must return at once, silently
        bench.barrier(w)
        out.put((r, w, lr, t, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_the_max_time_and_only_rank0_reports():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [(r, w, lr) for r, w, lr, _, _ in res] == [(0, 2, 0), (1, 2, 1)]
    assert all(t == 15.0 for *_, t, _ in res)          # max over ranks, on every rank
    assert res[1][4] == ""                              # rank 1 printed nothing


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
