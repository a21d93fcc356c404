"""The benchmark's multi-process plumbing on CPU: two `gloo` ranks read their
rank from the environment, meet at the barrier, agree on the maximum of their
timings, and the reference arm runs on rank 0 only (replicas only: there is
no data exchange between ranks)."""

import argparse
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        bench.barrier(w)
        m = bench.max_over_ranks(10.0 + 3.0 * rank, w)
        # the reference arm: rank 0 times the oracle, the others return at once
        skipped = None
        if rank != 0:
            skipped = bench.bench_reference(argparse.Namespace(workload="c1", steps=1, warmup=0)) is None
        q.put((rank, r, w, local, m, skipped))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(rank, 2, port, q)) for rank in range(2)]
    for p in procs:
        p.start()
    out = {}
    for _ in procs:
        rank, r, w, local, m, skipped = q.get(timeout=180)
        out[rank] = (r, w, local, m, skipped)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0][:3] == (0, 2, 0) and out[1][:3] == (1, 2, 1)
    assert out[0][3] == out[1][3] == 13.0  # max over ranks
    assert out[1][4] is True               # rank 1 does no reference work
