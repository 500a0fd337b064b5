"""Multi-process host logic for running the guided step on several GPUs.

The step is independent per sample: every output element depends only on the
same sample's inputs at the same position (and that sample's regional slabs),
so a batch shards by sample with no exchange on the data path.  The only
shared state is per run: the sigma schedule and the per-step scale table,
which every rank must hold identically.  The BCG write-up ("3. 张量并行下的
bucket构造" and edge case 3 of section 5) makes the same point for tensor
parallelism: the bucket table is broadcast once to every worker so that all
of them agree on bucket boundaries.

This module holds the host side of that: contiguous sample shards, the
one-time replication of the schedule and table from rank 0, and the
max-over-ranks reduction used for timing.  It works with any
``torch.distributed`` backend (NCCL on GPUs, gloo on CPU for tests).
"""

from __future__ import annotations

from typing import Optional, Tuple

import numpy as np


def shard_samples(B: int, rank: int, world: int) -> Tuple[int, int]:
    """Contiguous share of ``B`` samples for ``rank``: (first sample, count).

    Shares differ by at most one sample; lower ranks take the larger ones.
    """
    if world < 1 or not 0 <= rank < world or B < 0:
        raise ValueError("need 0 <= rank < world and B >= 0")
    base, extra = divmod(B, world)
    first = rank * base + min(rank, extra)
    return first, base + (1 if rank < extra else 0)


def replicate_plan(sigmas: Optional[np.ndarray], lut: Optional[np.ndarray], group=None,
                   device=None):
    """Broadcast rank 0's schedule (float32) and scale table (float32 or None).

    Every rank returns identical numpy arrays.  ``device`` is where the
    broadcast tensors live (a CUDA device for NCCL, CPU for gloo).
    """
    import torch
    import torch.distributed as dist

    dev = torch.device("cpu") if device is None else torch.device(device)
    rank = dist.get_rank(group)
    header = torch.zeros(2, dtype=torch.int64, device=dev)
    if rank == 0:
        header[0] = len(sigmas)
        header[1] = -1 if lut is None else len(lut)
    dist.broadcast(header, src=dist.get_global_rank(group, 0) if group is not None else 0,
                   group=group)
    n_sig, n_lut = int(header[0]), int(header[1])
    src = dist.get_global_rank(group, 0) if group is not None else 0
    sig_t = (torch.from_numpy(np.ascontiguousarray(sigmas, dtype=np.float32)).to(dev)
             if rank == 0 else torch.empty(n_sig, dtype=torch.float32, device=dev))
    dist.broadcast(sig_t, src=src, group=group)
    lut_out = None
    if n_lut >= 0:
        lut_t = (torch.from_numpy(np.ascontiguousarray(lut, dtype=np.float32)).to(dev)
                 if rank == 0 else torch.empty(n_lut, dtype=torch.float32, device=dev))
        dist.broadcast(lut_t, src=src, group=group)
        lut_out = lut_t.cpu().numpy()
    return sig_t.cpu().numpy(), lut_out


def max_over_ranks(value: float, group=None, device=None) -> float:
    """The largest ``value`` over the ranks of ``group`` (job time = slowest rank)."""
    import torch
    import torch.distributed as dist

    dev = torch.device("cpu") if device is None else torch.device(device)
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())
