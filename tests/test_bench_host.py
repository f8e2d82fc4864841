"""Host logic of the bench's multi-process path (replicas, no data-path
collective): two gloo ranks on CPU agree on the slowest rank's time and the
whole-job throughput."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    import sys
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    r, w, _ = bench.dist_setup()
    local_ms = 10.0 + 5.0 * r          # rank 1 is slower
    ms = bench.max_over_ranks(local_ms)
    value = bench.job_throughput(4000, w, ms / 1e3)
    bench.barrier()
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, w, ms, value))


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
    for r, w, ms, value in res:
        assert w == 2 and ms == 15.0
        assert value == pytest.approx(2 * 4000 / 0.015)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(100, 1, 0.5) == 200
