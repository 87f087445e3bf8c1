"""The bench's multi-rank path on CPU: two gloo ranks, as torchrun would start
them.  Replicas need no data exchange; what crosses ranks is the barrier and
the max over ranks of the timed duration, from which the whole-job rate is
the work of all replicas divided by the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, times, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        dist.barrier()
        t_max = bench.max_over_ranks(times[rank])
        rate = bench.aggregate_rate(w, 1.5e12, 10, t_max)
        q.put((r, w, local, t_max, rate))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(100.0, 125.0), (80.0, 40.0)])
def test_two_gloo_ranks_reduce_the_slowest_time(times):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    want_max = max(times)
    for r, (rank, world, local, t_max, rate) in enumerate(res):
        assert (rank, world, local) == (r, 2, r)
        assert t_max == want_max
        # two replicas x 10 steps x 1.5e12 units over the slowest rank's time
        assert rate == pytest.approx(2 * 10 * 1.5e12 / (want_max * 1e-3))


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.aggregate_rate(1, 2.0, 5, 1000.0) == pytest.approx(10.0)
