"""The multi-rank bench path on CPU: two gloo ranks over 127.0.0.1 (no GPU).  The job's step
time is the slowest rank's, every rank sees the same value, and under the reference arm only
rank 0 runs (the others return at once, without running the oracle)."""
import argparse
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.slowest(0.5 + rank, world, "cpu")
        ref = bench.run_reference(argparse.Namespace(steps=1, warmup=0), rank, world) if rank else 0
        dist.barrier()
        q.put((rank, t, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    for _ in procs:
        rank, t, ref = q.get(timeout=120)
        got[rank] = (t, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0][0] == got[1][0] == 1.5  # both ranks take the slowest rank's time
    assert got[1][1] is None               # the reference arm runs on rank 0 only


def test_one_rank_is_local():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest(0.25, 1, "cpu") == 0.25
