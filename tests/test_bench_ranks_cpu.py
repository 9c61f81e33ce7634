"""The multi-rank side of bench.py on the CPU (two gloo ranks): each rank runs its
own replica of the step, the step time is the slowest rank's, and the reported
throughput counts every rank's units."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = bench.max_over_ranks(times[rank], torch.device("cpu"), world)
        q.put((rank, ms, bench.job_rate(world, 1e9, ms)))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(240)
def test_two_ranks_take_the_slowest_time_and_count_both():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [3.0, 5.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=200) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [5.0, 5.0]
    # 2 ranks x 1e9 units per 5 ms step
    assert all(abs(o[2] - 2 * 1e9 / 5e-3) < 1e-3 for o in out)


def test_single_rank_is_unchanged():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, torch.device("cpu"), 1) == 7.5
    assert bench.job_rate(1, 2e12, 4.0) == 2e12 / 4e-3
