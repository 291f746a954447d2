"""Independent checkers used to pin the oracle (pure Python, small inputs only).

Nothing here calls the oracle or the CUDA library.  Each function restates a
definition directly -- enumeration of all alignments, scoring of a given CIGAR
-- so that a mistake in the oracle's dynamic programming shows up as a
disagreement.
"""
from __future__ import annotations

import itertools

OP_M, OP_I, OP_D = 0, 1, 2


def score_ops(ops, t, q, sub, o, e, start=(0, 0)):
    """Score of an alignment given as a list of ops, starting at cell ``start``.

    M consumes t_i and q_j and adds sub[t_i][q_j]; I consumes q_j; D consumes
    t_i; every maximal run of I (or of D) of length k costs o + k*e.
    Returns (score, i_end, j_end).
    """
    i, j = start
    s = 0
    prev = None
    for op in ops:
        if op == OP_M:
            s += int(sub[t[i]][q[j]])
            i += 1
            j += 1
        elif op == OP_I:
            s -= e + (o if prev != OP_I else 0)
            j += 1
        else:
            s -= e + (o if prev != OP_D else 0)
            i += 1
        prev = op
    return s, i, j


def runs_to_ops(runs):
    out = []
    for r in runs:
        out.extend([int(r) & 15] * (int(r) >> 4))
    return out


def rescore_cigar(runs, t, q, sub, o, e):
    return score_ops(runs_to_ops(runs), t, q, sub, o, e)


def all_paths(m, n, start=(0, 0)):
    """Every op sequence from ``start`` that stays inside [0..m] x [0..n]
    (the empty sequence included)."""
    out = []

    def rec(i, j, acc):
        out.append(tuple(acc))
        if i < m and j < n:
            acc.append(OP_M); rec(i + 1, j + 1, acc); acc.pop()
        if j < n:
            acc.append(OP_I); rec(i, j + 1, acc); acc.pop()
        if i < m:
            acc.append(OP_D); rec(i + 1, j, acc); acc.pop()

    rec(start[0], start[1], [])
    return out


def _rank(op, after):
    # preference when walking back from the end cell: after an I the walk
    # prefers leaving the gap (diagonal, then D) over extending it; elsewhere
    # diagonal > I > D
    if after == OP_I:
        return {OP_M: 0, OP_D: 1, OP_I: 2}[op]
    return {OP_M: 0, OP_I: 1, OP_D: 2}[op]


def backward_key(ops):
    key = []
    after = None
    for op in reversed(ops):
        key.append(_rank(op, after))
        after = op
    return tuple(key)


def brute_extend(t, q, sub, o, e):
    """Unpruned one-sided extension by enumeration of every alignment from the
    origin.  Returns (score, i_end, j_end, ops) with the end cell the earliest
    (smallest i+j, then smallest i) among maximal-score cells and ops the
    alignment preferred by the tie rule (diagonal > I > D, gap open > extend)."""
    m, n = len(t), len(q)
    paths = all_paths(m, n)
    scored = [(score_ops(p, t, q, sub, o, e), p) for p in paths]
    best = max(s for (s, _, _), _ in scored)
    ends = sorted({(i + j, i) for (s, i, j), _ in scored if s == best})
    d, i = ends[0]
    j = d - i
    cands = [p for (s, ii, jj), p in scored if s == best and ii == i and jj == j]
    chosen = min(cands, key=backward_key)
    return best, i, j, list(chosen)


def brute_local(t, q, sub, o, e):
    """Unpruned local alignment score with a zero floor by enumeration of all
    alignments from every start cell.  Returns (score, i_end, j_end) with the
    earliest (i+j, then i) cell among those reaching the maximum (the origin
    when nothing beats 0)."""
    m, n = len(t), len(q)
    cell_best = {(i, j): 0 for i in range(m + 1) for j in range(n + 1)}
    for i0, j0 in itertools.product(range(m + 1), range(n + 1)):
        for p in all_paths(m, n, (i0, j0)):
            if not p:
                continue
            s, i, j = score_ops(p, t, q, sub, o, e, (i0, j0))
            if s > cell_best[(i, j)]:
                cell_best[(i, j)] = s
    best = max(cell_best.values())
    d, i = min((i + j, i) for (i, j), s in cell_best.items() if s == best)
    return best, i, d - i
