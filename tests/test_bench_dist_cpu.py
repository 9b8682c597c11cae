"""The bench's multi-rank host logic on CPU: two ranks over gloo (127.0.0.1), as
torchrun would start them, agree on the slowest rank's time; the reference arm
works on rank 0 only."""
import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, secs, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    w, r, _ = bench.dist_setup(backend="gloo")
    q.put((r, w, bench.max_over_ranks(secs, w)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [0.125, 0.5]   # rank 1 is the slow one
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times[r], q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 for g in got)
    assert all(g[2] == max(times) for g in got)
    assert all(p.exitcode == 0 for p in procs)


def test_one_rank_needs_no_process_group():
    assert bench.max_over_ranks(0.25, 1) == 0.25


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class Args:
        steps, warmup = 1, 3
    bench.run_reference(Args(), 2, 1)   # rank 1 of 2: no work, no line
    assert capsys.readouterr().out == ""
