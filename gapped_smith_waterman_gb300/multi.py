"""Spreading one seed batch over several GPUs (one process per GPU).

Seed extensions are independent (FastZ, section 1: each seed extension can be
computed in parallel), so a batch shards by contiguous ranges of seeds with no
collective on the data path: every rank extends its range against its own
copy of the packed sequences and the per-rank results are concatenated in
rank order.  Only the final gather (and a timing max, in the benchmark)
communicates.
"""
from __future__ import annotations

import numpy as np


def shard_bounds(n_seeds: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous range [lo, hi) of seeds for ``rank``; ranges differ in size by
    at most one and cover 0 .. n_seeds-1 in rank order."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world size")
    base, extra = divmod(n_seeds, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo, hi


def rebase_cigars(results: np.ndarray, offset: int) -> np.ndarray:
    """Shift the CIGAR offsets of one rank's result records by ``offset`` runs
    (the position of that rank's CIGAR runs in the concatenated arena)."""
    out = results.copy()
    has = out["cigar_len"] > 0
    out["cigar_off"][has] += np.uint32(offset)
    return out


def gather_results(results: np.ndarray, cigar: np.ndarray, group=None):
    """All-gather per-rank (results, cigar) in rank order (torch.distributed,
    any backend that supports object collectives).  Returns the concatenated
    records, with CIGAR offsets rebased, and the concatenated CIGAR runs."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts = [None] * world
    dist.all_gather_object(parts, (results, cigar), group=group)
    recs, cigs, off = [], [], 0
    for res, cig in parts:
        recs.append(rebase_cigars(res, off))
        cigs.append(cig)
        off += int(cig.size)
    return np.concatenate(recs), (np.concatenate(cigs) if cigs else np.zeros(0, np.uint32))
