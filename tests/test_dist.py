"""Host-side logic of the multi-GPU benchmark (replicas, weak scaling) on two
gloo ranks on the CPU: the slowest rank's time is taken, the work of all
ranks is counted."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.0, 3.0][rank]  # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, dist, "cpu")
    value = bench.weak_scaling_value(4e9, world, worst)
    q.put((rank, worst, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, worst, value in results:
        assert worst == 3.0
        assert value == pytest.approx(4e9 * 2 / 3e-3 / 1e12)


def test_single_process_helpers():
    import bench
    assert bench.max_over_ranks(1.5) == 1.5
    assert bench.weak_scaling_value(1e12, 1, 1000.0) == pytest.approx(1.0)


def test_percentiles_nearest_rank():
    import bench
    assert bench.percentiles(list(range(1, 11))) == [1, 5, 9]
    assert bench.percentiles([3.0]) == [3.0, 3.0, 3.0]
    assert bench.percentiles([5, 1, 4, 2, 3], qs=(0, 100)) == [1, 5]
