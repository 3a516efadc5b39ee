"""The replica (N > 1) timing path of bench.py on CPU ranks over gloo:
every rank reports its own step time, the job time is the slowest rank's,
and the whole-job rate counts every rank's units."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_s = 0.010 * (rank + 1)            # rank 1 is the slow one
        job_s = bench.reduce_max(step_s, dist, "cpu")
        rate = bench.job_throughput(1000, world, job_s)
        dist.barrier()
        q.put((rank, job_s, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, job_s, rate in res:
        assert abs(job_s - 0.020) < 1e-12
        assert abs(rate - 2 * 1000 / 0.020) < 1e-6


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(0.5) == 0.5
    assert bench.job_throughput(10, 1, 2.0) == 5.0
