"""Helpers for the GPU parity tests: run a workload through the C ABI and
compare every field with the CPU oracle."""
from __future__ import annotations

import functools
import os

import numpy as np

from gapped_smith_waterman_gb300 import workloads as W

NTHREADS = max(1, (os.cpu_count() or 2))


@functools.lru_cache(maxsize=None)
def workload(cfg: int):
    return W.make(cfg)


def gpu_run(w, seeds=None, host=False):
    from gapped_smith_waterman_gb300 import fz
    ext = fz.Extender.for_workload(w)
    try:
        if host:
            res, cig = ext.extend_workload_host(w, seeds)
            return res, cig, None
        return ext.extend_workload(w, seeds)
    finally:
        ext.close()


def oracle_run(w, seeds=None, ydrop=None):
    import oracle
    return oracle.extend_batch(w, seeds=seeds, nthreads=NTHREADS, ydrop=ydrop)


def compare(w, seeds, gres, gcig, ores, ocig, ooff, check_cigar=True, label=""):
    """Bit-exact comparison of score, end cell, CIGAR (genomic order) and flags."""
    seeds = w.seeds if seeds is None else seeds
    n = len(seeds)
    side = seeds["side"].astype(np.int64)
    req = np.zeros(2 * n, bool)
    req[0::2] = (side & 1) != 0
    req[1::2] = (side & 2) != 0
    g_done = (gres["flags"] & 1) != 0
    assert np.array_equal(g_done, req), f"{label}: requested flags differ"
    for f_g, f_o in (("score", "score"), ("t_end", "i_end"), ("q_end", "j_end")):
        bad = np.flatnonzero(gres[f_g] != ores[f_o])
        assert bad.size == 0, (f"{label}: {f_g} differs at {bad.size} extensions, first x={bad[0]}: "
                               f"gpu {gres[bad[0]]} oracle {ores[bad[0]]}")
    eager = (gres["flags"] & 2) != 0
    corner = (ores["i_end"] <= 16) & (ores["j_end"] <= 16) & req
    wide = (gres["flags"] & 4) != 0
    assert np.array_equal(eager & ~wide, corner & ~wide), f"{label}: eager flag mismatch"
    if not check_cigar or w.mode != W.MODE_EXTEND:
        return
    for x in np.flatnonzero(req):
        o = ores[x]
        runs_o = ocig[ooff[x]:ooff[x] + o["n_cigar"]]
        if x & 1:
            runs_o = runs_o[::-1]
        g = gres[x]
        runs_g = gcig[g["cigar_off"]:g["cigar_off"] + g["cigar_len"]]
        assert np.array_equal(runs_g, runs_o), (f"{label}: CIGAR differs at x={x}: gpu {runs_g[:12]} "
                                                f"oracle {runs_o[:12]}")


def sample_seeds(w, k, seed=0):
    rng = np.random.default_rng(seed)
    idx = np.sort(rng.choice(len(w.seeds), size=min(k, len(w.seeds)), replace=False))
    return idx


def sub_workload(w, idx):
    return W.Workload(w.name, w.target, w.query, w.seeds[idx], w.sub, w.gap_open, w.gap_extend, w.ydrop,
                      w.max_len, w.mode, w.note)
