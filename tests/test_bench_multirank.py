"""bench.py's multi-rank plumbing on CPU: two gloo ranks, max-over-ranks timing
and the barrier, as torchrun would launch them (replicas, no data-path
collective)."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        t = bench.max_over_ranks(0.5 + rank, world)   # rank 1 is the slowest
        q.put((rank, t))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 1.5, 1: 1.5}


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_step_bytes_of_the_128k_workload():
    sys.path.insert(0, ROOT)
    import bench
    import synth
    import numpy as np
    p = synth.Params(num_q_heads=32, initial_blocks=1, local_blocks=32, top_k=32,
                     rep=synth.REP_QUEST, head_mode=synth.HEAD_SHARED)
    pool = np.empty((0, 8, 128, 128), dtype=np.uint16)  # shapes only
    w = synth.Workload("shape-only", 0, pool, pool, np.zeros((1, 1024), np.int32),
                       np.array([131072], np.int32), np.empty((1, 32, 128), np.uint16), p)
    b = bench.step_bytes(w)
    assert b["reps"] == 991 * 8 * 2 * 256          # 4.06 MB
    assert b["kv"] == (128 + 32 * 128 + 4096) * 8 * 512  # 34.08 MB
