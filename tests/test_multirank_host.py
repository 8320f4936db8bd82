"""Host side of the multi-GPU bench path, as two gloo ranks on the CPU.

Tokens are independent and routing is static, so ranks share the tables and weights and
each takes its own batch ("weak" scaling); the only exchange is the timing reduction:
the job's time is the slowest rank's, and its rate counts every rank's tokens.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import l3_workloads as W

        local_ms = [3.0, 5.0][rank]  # rank 1 is the slow one
        total = bench.max_over_ranks(local_ms, "cpu")
        wl = W.make(2, T=256, shard=rank)
        out.put((rank, total, bench.job_rate(world, wl.T, 10, total), wl.ids.tobytes(),
                 wl.W_up.tobytes(), wl.table_seed))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_take_the_slowest_time_and_own_batches():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        r, total, rate, ids, w_up, seed = out.get(timeout=240)
        res[r] = (total, rate, ids, w_up, seed)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest rank's time and the same whole-job rate
    assert res[0][0] == res[1][0] == 5.0
    assert res[0][1] == res[1][1] == pytest.approx(2 * 256 * 10 / 5e-3)
    # each rank draws its own batch, over the same weights and tables
    assert res[0][2] != res[1][2]
    assert res[0][3] == res[1][3] and res[0][4] == res[1][4]


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.5, "cpu") == 7.5
    assert bench.job_rate(1, 8192, 20, 4.0) == pytest.approx(8192 * 20 / 4e-3)
    assert np.isfinite(bench.job_rate(8, 1, 1, 1.0))
