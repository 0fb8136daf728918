"""The bench's replica bookkeeping over two CPU ranks (gloo): the timings reported are the maximum
over the ranks; the per-step time stays one rank's and the job's step rate counts every replica."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, root, q):
    import sys

    try:
        sys.path.insert(0, root)
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import bench

        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.25 * (rank + 1)], world, "cpu")
        q.put((rank, got, bench.replica_step_rates(got[0], world)))
        dist.barrier()
        dist.destroy_process_group()
    except Exception as e:  # report instead of leaving the parent waiting
        q.put((rank, repr(e), None))


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, root, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, got, job in results:
        assert got == [2.0, 10.0, 0.5]
        us, rate = job
        assert us == pytest.approx(2000.0)  # the slowest rank's 2 ms step, not divided by N
        assert rate == pytest.approx(1000.0)  # two replica steps every 2 ms


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks([3.0, 4.0], 1, "cpu") == [3.0, 4.0]
    us, rate = bench.replica_step_rates(0.25, 1)
    assert us == pytest.approx(250.0) and rate == pytest.approx(4000.0)
    assert torch.distributed.is_initialized() is False
