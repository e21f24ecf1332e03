"""The benchmark's multi-replica timing on CPU: two gloo ranks, each with its
own step time, must both see the slowest rank's time, and the job rate must
count every replica's tokens.  The step itself has no exchange between
ranks (replicas only), so this is the whole of the N > 1 path."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, results):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank])
        results[rank] = (ms, bench.job_tokens_per_s(1000, world, 10, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_with_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    world, port = 2, _free_port()
    times = [3.5, 5.25]
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, times, results))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0, 0], codes
        got = dict(results)
    for r in range(world):
        ms, rate = got[r]
        assert ms == 5.25
        assert rate == pytest.approx(1000 * 2 * 10 / 5.25e-3)


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.0) == 2.0
    assert bench.job_tokens_per_s(512 * 8, 1, 4, 2.0) == pytest.approx(512 * 8 * 4 / 2e-3)
