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


def test_ablation_overrides():
    import argparse
    import bench
    ns = argparse.Namespace(workload="llama7b_x8_sample", tokens=0, alpha=None, X="4,32", no_decs=True)
    wl = bench._workload(ns)
    assert wl.X == [4, 32] and wl.decs is False


def test_reference_arm_line_matches_the_library_line(capsys):
    """The oracle arm decodes the same unit from a prefilled prompt and prints the library
    line's config keys and e2e unit (so the two lines compare)."""
    import argparse
    import json
    import bench
    args = argparse.Namespace(workload="tiny", tokens=4, alpha=None, X=None, no_decs=False, ar=False,
                              max_branch=0, adapters=None, steps=1, warmup=0)
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "committed tokens/s"
    assert line["e2e"]["unit"] == line["unit"] and line["value"] > 0
    wl = bench._workload(args)
    assert line["config"] == json.loads(json.dumps(bench._config(args, wl, 1, wl.batch)))
    assert "prefill" in line["cpu_baseline"]["sample"]


def test_one_core_block_restores_affinity():
    import os
    import bench
    before = os.sched_getaffinity(0)
    with bench._OneCore():
        assert len(os.sched_getaffinity(0)) == 1
    assert os.sched_getaffinity(0) == before


def test_prefill_flop_count():
    """The bench's prefill FLOP count, checked by brute force on a tiny shape: every linear
    layer's 2 FLOP per weight and position, and 4 * head_dim FLOP per (query head, query,
    visible key) pair counted one pair at a time."""
    sys.path.insert(0, ROOT)
    import bench
    import dex_inputs as di
    shape = di.ModelShape(n_layers=3, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64, d_ff=512,
                          vocab=1000, tied_head=False)
    B, P = 2, 7
    weights = (4 * 64 + 2 * 2 * 64) * 256 + 4 * 64 * 256 + 3 * 512 * 256   # QKV, O, gate/up/down
    linear = 2 * weights * P
    attn = sum(4 * 64 * 4 for q in range(P) for k in range(q + 1))
    assert bench.prefill_flop(shape, B, P) == B * 3 * (linear + attn)
    # the 7B-shaped prompt of the benchmark: about 6.9 TFLOP (the weights dominate)
    assert 6.5e12 < bench.prefill_flop(di.LLAMA7B, 1, 511) < 7.2e12
