"""The multi-replica path of bench.py on CPU: two gloo ranks agree on the
slowest rank's step time and on the whole-job throughput."""
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


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    bench.barrier(w)
    step_ms = 10.0 + 5.0 * r                      # rank 1 is slower
    value, ms = bench.aggregate(2.0e9, step_ms, w)
    q.put((r, w, lr, value, ms))
    dist.destroy_process_group()


def test_two_replicas_aggregate_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, lr, value, ms in res:
        assert w == 2 and lr == r
        assert ms == 15.0                          # the slowest rank's step time
        assert value == pytest.approx(2 * 2.0e9 / 15e-3 / 1e9)


def test_single_process_aggregate():
    import bench
    value, ms = bench.aggregate(1.0e9, 4.0, 1)
    assert ms == 4.0 and value == pytest.approx(250.0)
