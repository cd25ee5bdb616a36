"""The multi-GPU path is replicas only: every rank runs an independent decode and the job's
throughput is all ranks' bytes over the slowest rank's time.  This checks that aggregation
with two gloo ranks on CPU (no GPU, no data-path collective)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, ms, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    res = bench.job_throughput(ms[rank], 1e9, world, torch.device("cpu"))
    q.put((rank, res))
    dist.barrier()
    dist.destroy_process_group()


def test_job_throughput_takes_the_slowest_rank():
    world, port = 2, _free_port()
    ms = {0: [2.0, 5.0], 1: [4.0, 3.0]}   # per-rank (device step, end-to-end) times in ms
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, ms, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        (v0, m0), (v1, m1) = out[r]
        assert m0 == 4.0 and m1 == 5.0                      # max over ranks, per timing
        assert v0 == pytest.approx(2 * 1e9 / 4e-3 / 1e9)    # both ranks' bytes / slowest time
        assert v1 == pytest.approx(2 * 1e9 / 5e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    (v, m), = bench.job_throughput([2.0], 1e9, 1, torch.device("cpu"))
    assert m == 2.0 and v == pytest.approx(500.0)
