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


def _dcp_rank(rank: int, world: int, port: int, out):
    """One context-parallel rank: its shard's partial by the oracle, an
    all-gather of (O, LSE) over gloo, then the log-sum-exp merge."""
    import numpy as np
    import oracle
    from tests import pins
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(5)          # same problem on every rank
        P = pins.Paged(rng, 8, 2, 16, 4, [1, 1, 2], [37, 9, 50], q_scale=2.0)
        o, lse = P.run(None, shard=(world, rank, 4))
        o_t, l_t = torch.from_numpy(o), torch.from_numpy(lse)
        all_o = [torch.empty_like(o_t) for _ in range(world)]
        all_l = [torch.empty_like(l_t) for _ in range(world)]
        dist.all_gather(all_o, o_t)
        dist.all_gather(all_l, l_t)
        merged = np.stack([oracle.lse_merge(np.array([l[r].item() for l in all_l]),
                                            np.stack([x[r].numpy() for x in all_o]))[0]
                           for r in range(o.shape[0])])
        full, _ = P.run(None)
        out.put((rank, float(np.abs(merged - full).max())))
    finally:
        dist.destroy_process_group()


def test_dcp_exchange_and_merge_on_two_gloo_ranks():
    """Decode context parallelism's exchange step (page "vLLM Agentic 推理",
    section 4.3.3, steps 3-4) on two CPU ranks: each rank's partial over its
    own tokens, gathered and merged, is the unsharded attention."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dcp_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _ in res] == [0, 1]
    assert all(err < 1e-12 for _, err in res), res
