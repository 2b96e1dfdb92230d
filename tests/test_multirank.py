"""The multi-process path of bench.py on CPU: two ranks over gloo (127.0.0.1), as torchrun would
launch them on two GPUs.  The path has no data exchange (replicas only); what the ranks share is
the timing: every rank must see the slowest rank's time, and the job's value counts the units of
every rank over that time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], dist, device="cpu")
        value = bench.job_value(dist.get_world_size(), 1000.0, ms / 1e3)
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_two_ranks_share_the_slowest_time():
    world, port = 2, _free_port()
    times = [3.5, 7.25]   # ms per rank
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1], "ranks disagree on the job's time"
    ms, value = res[0]
    assert ms == max(times)
    # 2 ranks x 1000 units over the slowest rank's 7.25 ms
    assert value == pytest.approx(2 * 1000.0 / 7.25e-3)


def test_single_process_needs_no_collective():
    import bench
    assert bench.max_over_ranks(4.0, None) == 4.0
    assert bench.job_value(1, 500.0, 0.5) == 1000.0
