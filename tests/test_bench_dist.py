"""The multi-process path of bench.py on CPU: two ranks over gloo (world size 2).

The hot path shards by batch / head group with no exchange, so bench.py runs one replica per
rank ("weak" scaling). What needs checking without GPUs is the plumbing: process-group setup
from the torchrun environment, the barrier, the max-over-ranks step time, the whole-job rate,
and that only rank 0 runs the reference arm.
"""
import argparse
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    try:
        import bench

        r, w, local, pg = bench.dist_setup(world)
        bench.barrier(pg)
        step_ms = 1.5 * (r + 1)  # rank 1 is the slow one
        mx = bench.max_over_ranks(pg, step_ms)
        rate = bench.aggregate_tflops(2.0e12, w, mx)
        ref_skipped = bench.bench_reference(argparse.Namespace(steps=1, warmup=3), r, w) is None if r != 0 else None
        bench.barrier(pg)
        pg.destroy_process_group()
        q.put((r, w, local, mx, rate, ref_skipped, None))
    except Exception as e:  # reported to the parent
        q.put((rank, None, None, None, None, None, repr(e)))


def test_two_rank_gloo_plumbing():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = {}
    for _ in procs:
        r, w, local, mx, rate, ref_skipped, err = q.get(timeout=180)
        assert err is None, err
        results[r] = (w, local, mx, rate, ref_skipped)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(results) == [0, 1]
    for r, (w, local, mx, rate, ref_skipped) in results.items():
        assert w == 2 and local == r
        assert mx == pytest.approx(3.0)  # the max over ranks, seen by every rank
        # two replicas of 2 TFLOP each in 3 ms
        assert rate == pytest.approx(2 * 2.0e12 / 3.0e-3 / 1e12)
    assert results[1][4] is True  # rank 1 does not run the reference arm


def test_aggregate_single_rank():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.aggregate_tflops(3.0e12, 1, 1.0) == pytest.approx(3000.0)
