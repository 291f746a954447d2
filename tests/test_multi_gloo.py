"""Host logic of the sharded (one process per GPU) path, on CPU with gloo.

Two ranks each extend a contiguous shard of one seed batch and all-gather the
records; the gathered batch must equal the unsharded one record for record,
CIGAR runs included.  The per-rank extension here is the oracle (the CPU has
no GPU); what is under test is the shard split, the CIGAR-offset rebasing and
the rank-order gather.
"""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from gapped_smith_waterman_gb300 import fz, workloads
from gapped_smith_waterman_gb300.multi import gather_results, rebase_cigars, shard_bounds


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _as_records(w, seeds):
    """Oracle output for ``seeds`` in the library's record layout: one packed
    CIGAR arena, cigar_off/cigar_len per extension (right, left per seed)."""
    res, cig, off = oracle.extend_batch(w, seeds=seeds, nthreads=2)
    out = np.zeros(res.size, fz.RESULT_DTYPE)
    runs, pos = [], 0
    for x in range(res.size):
        k = int(res["n_cigar"][x])
        out["score"][x] = res["score"][x]
        out["t_end"][x] = res["i_end"][x]
        out["q_end"][x] = res["j_end"][x]
        out["cigar_len"][x] = k
        out["cigar_off"][x] = pos if k else 0
        runs.append(cig[off[x]:off[x] + k])
        pos += k
    return out, (np.concatenate(runs).astype(np.uint32) if runs else np.zeros(0, np.uint32))


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = workloads.make_cfg1(n_pairs=37)
        lo, hi = shard_bounds(len(w.seeds), rank, world)
        rec, cig = _as_records(w, w.seeds[lo:hi])
        g_rec, g_cig = gather_results(rec, cig)
        q.put((rank, g_rec.tobytes(), g_cig.tobytes()))
    finally:
        dist.destroy_process_group()


def test_shard_bounds_cover():
    for n in (0, 1, 7, 8, 100, 1001):
        for world in (1, 2, 3, 8):
            spans = [shard_bounds(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            for (a, b), (c, d) in zip(spans, spans[1:]):
                assert b == c
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_bounds(10, 2, 2)


def test_rebase_skips_empty():
    rec = np.zeros(3, fz.RESULT_DTYPE)
    rec["cigar_len"] = [2, 0, 1]
    rec["cigar_off"] = [0, 0, 2]
    out = rebase_cigars(rec, 10)
    assert list(out["cigar_off"]) == [10, 0, 12]
    assert list(rec["cigar_off"]) == [0, 0, 2]


def test_gloo_two_ranks_gather_equals_unsharded():
    oracle.build()
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = workloads.make_cfg1(n_pairs=37)
    ref_rec, ref_cig = _as_records(w, w.seeds)
    for rank, rec_b, cig_b in got:
        rec = np.frombuffer(rec_b, fz.RESULT_DTYPE)
        cig = np.frombuffer(cig_b, np.uint32)
        assert np.array_equal(rec, ref_rec), f"rank {rank}: records differ"
        assert np.array_equal(cig, ref_cig), f"rank {rank}: CIGAR arena differs"
