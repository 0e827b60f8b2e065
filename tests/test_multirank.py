"""The multi-GPU path of the benchmark is replicas: each rank runs its own batch
and caches, and the only exchange is the timing (the slowest rank's time sets
the job's).  Checked with two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r took (r+1) ms and 2(r+1) s; everyone must see the slowest rank's numbers
    ms, e2e = bench.max_over_ranks([1.0 + rank, 2.0 * (rank + 1)])
    q.put((rank, ms, e2e, bench.job_throughput(world, 4, 50, ms / 1000.0)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank_and_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, e2e, qps in out:
        assert ms == 2.0 and e2e == 4.0
        assert qps == pytest.approx(2 * 4 * 50 / 0.002)
