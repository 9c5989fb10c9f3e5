"""The multi-process path of bench.py on CPU: two ranks over gloo.

Each rank runs the same per-GPU workload (replicas); the ranks meet only for
the timing barrier and the max-over-ranks of the elapsed time, and `value`
is the units of all ranks over that time.  These tests run that plumbing in
world-size-2 gloo process groups (no GPU): the environment parsing, the
process group, the barrier, the max reduction, the whole-job rate, and the
reference arm's rule that ranks other than 0 exit without work.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    got_ws, got_rank, local = bench.dist_env()
    dist = bench.init_dist(got_ws, local)
    try:
        assert dist is not None and dist.get_backend() == "gloo"
        bench.barrier(dist)
        # each rank's elapsed time differs; all must see the maximum
        mx = bench.max_over_ranks(10.0 + 5.0 * rank, dist)
        rate = bench.job_rate(2.0e12, mx, got_ws, 1e12)
        # the reference arm: only rank 0 works; others return 0 at once
        class _A:
            gpus, steps, warmup = ws, 1, 3
        ref_rc = bench.reference_arm(_A()) if rank != 0 else None
        bench.barrier(dist)
        q.put((got_rank, got_ws, local, mx, rate, ref_rc))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_the_max_and_the_job_rate():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(ws))
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 and r[2] == r[0] for r in res)
    # both ranks see the slower rank's 15 ms; 2 ranks x 2e12 flops in 15 ms
    assert all(r[3] == 15.0 for r in res)
    assert all(abs(r[4] - 2 * 2.0e12 / 15e-3 / 1e12) < 1e-9 for r in res)
    assert res[1][5] == 0


def test_single_process_has_no_group():
    import bench
    assert bench.init_dist(1, 0) is None
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.job_rate(1e9, 2.0, 1, 1e9) == pytest.approx(500.0)
