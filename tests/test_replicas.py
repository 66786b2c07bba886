"""bench.py's replica path with world_size 2 on CPU (gloo): max-over-ranks timing and the
whole-job throughput.  The path needs no data exchange between GPUs; only the timing is reduced."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    times = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5 * (rank + 1)])
    results[rank] = (times, bench.job_gbs(1_000_000_000, world, times[0]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(2):
            times, gbs = results[r]
            assert times == [2.0, 10.0, 1.0]              # slowest rank wins every timing
            assert gbs == pytest.approx(2 * 1e9 / 2e-3 / 1e9)   # both ranks' bytes over the max time


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.job_gbs(2_000_000_000, 1, 1.0) == pytest.approx(2000.0)
