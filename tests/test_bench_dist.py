"""Multi-process aggregation of the benchmark (replicas only): two gloo ranks on CPU.

Each rank decodes its own request stream; the job's throughput is all ranks' committed
tokens over the slowest rank's time, and the barrier releases every rank together.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cpu = torch.device("cpu")
        tokens = [256.0, 128.0][rank]
        seconds = [2.0, 4.0][rank]
        v = bench.replica_throughput(tokens, seconds, world, cpu)
        m = bench.reduce_over_ranks(float(rank + 1), "max", world, cpu)
        s = bench.reduce_over_ranks(float(rank + 1), "sum", world, cpu)
        bench.rank_barrier(world)
        q.put((rank, v, m, s))
    finally:
        dist.destroy_process_group()


def test_two_rank_replica_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, v, m, s in res:
        assert v == pytest.approx((256.0 + 128.0) / 4.0)   # tokens of both ranks / slowest rank
        assert m == 2.0 and s == 3.0


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(3.5, "max", 1, None) == 3.5
    assert bench.replica_throughput(100.0, 2.0, 1, None) == 50.0


def test_workload_overrides():
    """--tokens and --alpha replace only their own fields of the named workload."""
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    base = bench._workload(argparse.Namespace(workload="llama7b_x8_sample", tokens=0, alpha=None))
    wl = bench._workload(argparse.Namespace(workload="llama7b_x8_sample", tokens=32, alpha=0.1))
    assert (wl.max_new, wl.alpha) == (32, 0.1)
    assert (base.max_new, base.alpha) == (256, 0.05)
    assert (wl.X, wl.tau, wl.sample, wl.shape) == (base.X, base.tau, base.sample, base.shape)
