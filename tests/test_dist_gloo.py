"""Multi-rank host logic on CPU: two gloo ranks (no GPU).

Checks the sample sharding (complete, disjoint, balanced), the one-time
replication of the schedule and bucket table from rank 0 (every rank ends with
rank 0's bits even when its own copy differs), and the max-over-ranks timing.
"""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from bucketized_guidance_step_gb300 import dist as D


@pytest.mark.parametrize("B,world", [(16, 2), (17, 2), (3, 4), (0, 3), (64, 8), (5, 1)])
def test_shards_cover_batch_once(B, world):
    seen = []
    sizes = []
    for r in range(world):
        first, n = D.shard_samples(B, r, world)
        seen.extend(range(first, first + n))
        sizes.append(n)
    assert seen == list(range(B))
    assert max(sizes) - min(sizes) <= 1


def test_shard_rejects_bad_rank():
    with pytest.raises(ValueError):
        D.shard_samples(4, 2, 2)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        if rank == 0:
            sig = np.array([14.6, 7.0, 2.5, 0.0], dtype=np.float32)
            lut = np.array([1.95, 1.85, 1.75], dtype=np.float32)
        else:                                     # a stale, different copy
            sig = np.array([1.0, 0.0], dtype=np.float32)
            lut = None
        got_sig, got_lut = D.replicate_plan(sig, lut)
        slowest = D.max_over_ranks(1.5 + rank)
        first, n = D.shard_samples(16, rank, world)
        q.put((rank, got_sig.tolist(), None if got_lut is None else got_lut.tolist(),
               slowest, first, n))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicate_and_reduce():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(2):
        r = q.get(timeout=120)
        results[r[0]] = r
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want_sig = np.array([14.6, 7.0, 2.5, 0.0], dtype=np.float32).tolist()
    want_lut = np.array([1.95, 1.85, 1.75], dtype=np.float32).tolist()
    for r in (0, 1):
        _, sig, lut, slowest, first, n = results[r]
        assert sig == want_sig and lut == want_lut
        assert slowest == 2.5
        assert (first, n) == ((0, 8) if r == 0 else (8, 8))
