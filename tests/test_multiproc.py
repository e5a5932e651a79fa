"""The multi-rank path of bench.py on CPU: two gloo ranks (127.0.0.1), as the
launcher runs them with one process per GPU. The decode path has no exchange
step, so ranks are replicas; what ranks share is the timing: the slowest
rank's time per step, and the whole-job throughput built from it."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 1.0 + rank * 0.5                      # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms, "cpu")
    value = bench.whole_job_gbs(6.0e8, slowest, world)
    q.put((rank, slowest, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_share_the_slowest_time_and_sum_the_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in results:
        assert slowest == pytest.approx(1.5)
        # 2 ranks x 0.6 GB per step / 1.5 ms = 800 GB/s
        assert value == pytest.approx(800.0)


def test_single_process_is_its_own_max():
    import bench
    assert bench.max_over_ranks(2.5, "cpu") == 2.5
    assert bench.whole_job_gbs(1e9, 1.0, 1) == pytest.approx(1000.0)
