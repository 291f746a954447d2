"""Canonical digests of seed-extension results, for comparing a large batch
against stored oracle results without storing every record.

This module holds no alignment arithmetic: it serialises result fields that
either side produced and hashes them.  For one-sided extension x = 2 k + side
(side 0 right, 1 left) the serialised form is the int32 quadruple (score,
t_end, q_end, number of CIGAR runs), then, after all quadruples of a chunk,
the chunk's CIGAR runs (uint32 ``(len << 4) | op``) in forward genomic order,
extension by extension.  Only hashes are compared: equal digests mean equal
records (up to a SHA-256 collision).
"""
from __future__ import annotations

import hashlib

import numpy as np

from gapped_smith_waterman_gb300 import workloads as W


def input_sha256(w) -> str:
    """Hash of everything a batch's results depend on: the packed sequences,
    the seed records and the scoring parameters."""
    h = hashlib.sha256()
    for a in (W.pack2(w.target), W.pack2(w.query), np.ascontiguousarray(w.seeds).view(np.uint8),
              np.ascontiguousarray(np.asarray(w.sub, np.int32))):
        h.update(np.ascontiguousarray(a).tobytes())
    h.update(np.array([w.gap_open, w.gap_extend, w.ydrop, w.max_len, w.mode], np.int64).tobytes())
    return h.hexdigest()


def chunk_digest(score, t_end, q_end, lens, runs) -> str:
    """score, t_end, q_end, lens: per extension of the chunk (lens = CIGAR
    runs); runs: the chunk's runs concatenated in extension order, each
    extension's in forward genomic order."""
    head = np.stack([np.asarray(score, np.int64), np.asarray(t_end, np.int64), np.asarray(q_end, np.int64),
                     np.asarray(lens, np.int64)], 1)
    h = hashlib.sha256()
    h.update(head.astype("<i4").tobytes())
    runs = np.asarray(runs, np.uint32)
    assert runs.size == int(np.asarray(lens, np.int64).sum())
    if runs.size:
        h.update(runs.astype("<u4").tobytes())
    return h.hexdigest()


def oracle_chunk(ores, ocig, ooff):
    """Fields of an oracle batch (oracle.extend_batch) in digest form."""
    parts = []
    for x in range(len(ores)):
        r = ocig[ooff[x]:ooff[x] + ores["n_cigar"][x]]
        parts.append(r[::-1] if x & 1 else r)      # left windows are walked backwards
    runs = np.concatenate(parts) if parts else np.zeros(0, np.uint32)
    return ores["score"], ores["i_end"], ores["j_end"], ores["n_cigar"], runs


def packed_chunk(res, packed, x0, x1):
    """Fields of extensions [x0, x1) from the host entry's records and its
    packed runs (extension x's runs at res[x].cigar_off, in extension order)."""
    g = res[x0:x1]
    lens = g["cigar_len"].astype(np.int64)
    if x1 > x0 and lens.sum():
        a = int(g["cigar_off"][0])
        assert np.array_equal(g["cigar_off"].astype(np.int64) - a, np.concatenate([[0], np.cumsum(lens)[:-1]]))
        runs = packed[a:a + int(lens.sum())]
    else:
        runs = np.zeros(0, np.uint32)
    return g["score"], g["t_end"], g["q_end"], lens, runs
