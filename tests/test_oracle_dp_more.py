"""Pins of the oracle's edit distance and dynamic time warping (the DPX
intrinsics article, section 1.3) against formulations other than its own
row-by-row table: brute force on tiny inputs, closed forms and invariants."""
import functools
import itertools

import numpy as np
import pytest

import oracle


def _edit_brute(a, b):
    """Levenshtein distance as a recursion from the end of both strings."""
    a, b = tuple(int(x) for x in a), tuple(int(x) for x in b)

    @functools.lru_cache(maxsize=None)
    def f(i, j):
        if i == 0:
            return j
        if j == 0:
            return i
        return min(f(i - 1, j) + 1, f(i, j - 1) + 1, f(i - 1, j - 1) + (a[i - 1] != b[j - 1]))
    return f(len(a), len(b))


def _edit_alignments(a, b):
    """Minimum over every alignment of a and b (each column a match/substitution,
    an insertion or a deletion) enumerated explicitly: tiny inputs only."""
    best = None
    m, n = len(a), len(b)

    def walk(i, j, cost):
        nonlocal best
        if best is not None and cost >= best:
            return
        if i == m and j == n:
            best = cost
            return
        if i < m and j < n:
            walk(i + 1, j + 1, cost + (a[i] != b[j]))
        if i < m:
            walk(i + 1, j, cost + 1)
        if j < n:
            walk(i, j + 1, cost + 1)
    walk(0, 0, 0)
    return best


def _dtw_paths(x, y):
    """Minimum over every monotone warping path from (1,1) to (m,n) with steps
    (1,0), (0,1), (1,1) of the summed |x_i - y_j| of its cells."""
    m, n = len(x), len(y)
    if m == 0 and n == 0:
        return 0
    if m == 0 or n == 0:
        return -1
    best = None

    def walk(i, j, cost):
        nonlocal best
        cost += abs(int(x[i]) - int(y[j]))
        if i == m - 1 and j == n - 1:
            best = cost if best is None else min(best, cost)
            return
        if i + 1 < m and j + 1 < n:
            walk(i + 1, j + 1, cost)
        if i + 1 < m:
            walk(i + 1, j, cost)
        if j + 1 < n:
            walk(i, j + 1, cost)
    walk(0, 0, 0)
    return best


def test_edit_distance_brute_force_on_tiny_strings():
    rng = np.random.default_rng(5)
    for _ in range(400):
        a = rng.integers(0, 4, int(rng.integers(0, 8))).astype(np.uint8)
        b = rng.integers(0, 4, int(rng.integers(0, 8))).astype(np.uint8)
        want = _edit_brute(a, b)
        assert oracle.edit_distance(a, b) == want
        if len(a) + len(b) <= 9:
            assert _edit_alignments(a, b) == want


def test_edit_distance_closed_forms_and_invariants():
    rng = np.random.default_rng(6)
    for _ in range(50):
        a = rng.integers(0, 4, int(rng.integers(1, 300))).astype(np.uint8)
        b = rng.integers(0, 4, int(rng.integers(1, 300))).astype(np.uint8)
        c = rng.integers(0, 4, int(rng.integers(1, 300))).astype(np.uint8)
        assert oracle.edit_distance(a, a) == 0
        assert oracle.edit_distance(a, []) == len(a) == oracle.edit_distance([], a)
        d = oracle.edit_distance(a, b)
        assert d == oracle.edit_distance(b, a)
        assert abs(len(a) - len(b)) <= d <= max(len(a), len(b))
        assert oracle.edit_distance(a, c) <= d + oracle.edit_distance(b, c)
        # one substitution: exactly 1; one base removed: exactly 1
        s = a.copy()
        k = int(rng.integers(0, len(a)))
        s[k] = (s[k] + 1) % 4
        assert oracle.edit_distance(a, s) == 1
        assert oracle.edit_distance(a, np.delete(a, k)) == 1
    # a homopolymer against another: every column a substitution or a gap
    assert oracle.edit_distance(np.zeros(7, np.uint8), np.ones(5, np.uint8)) == 7


def test_dtw_brute_force_on_tiny_sequences():
    rng = np.random.default_rng(7)
    for _ in range(300):
        x = rng.integers(-20, 21, int(rng.integers(0, 6))).astype(np.int32)
        y = rng.integers(-20, 21, int(rng.integers(0, 6))).astype(np.int32)
        assert oracle.dtw(x, y) == _dtw_paths(x, y)


def test_dtw_closed_forms_and_invariants():
    rng = np.random.default_rng(8)
    for _ in range(50):
        x = rng.integers(-1000, 1001, int(rng.integers(1, 200))).astype(np.int32)
        y = rng.integers(-1000, 1001, int(rng.integers(1, 200))).astype(np.int32)
        assert oracle.dtw(x, x) == 0
        d = oracle.dtw(x, y)
        assert d == oracle.dtw(y, x)
        # both ends are on every path
        assert d >= abs(int(x[0]) - int(y[0])) + (abs(int(x[-1]) - int(y[-1])) if len(x) + len(y) > 2 else 0)
        # repeating a sample costs nothing when it warps onto itself
        assert oracle.dtw(x, np.repeat(x, 2)) == 0
    for c1, c2, m, n in itertools.product((3, -7), (0, 11), (1, 4), (2, 9)):
        assert oracle.dtw(np.full(m, c1, np.int32), np.full(n, c2, np.int32)) == max(m, n) * abs(c1 - c2)
    assert oracle.dtw([], []) == 0 and oracle.dtw([], [1]) == -1 and oracle.dtw([1], []) == -1


@pytest.mark.parametrize("fn", ["edit", "dtw"])
def test_pairs_batch_reads_the_pair_slices(fn):
    rng = np.random.default_rng(9)
    a = rng.integers(0, 4, 500).astype(np.uint8) if fn == "edit" else rng.integers(-50, 50, 500).astype(np.int32)
    b = rng.integers(0, 4, 600).astype(np.uint8) if fn == "edit" else rng.integers(-50, 50, 600).astype(np.int32)
    pairs = np.zeros(6, [("a_pos", "<u8"), ("b_pos", "<u8"), ("a_len", "<u4"), ("b_len", "<u4")])
    pairs["a_pos"] = [0, 10, 100, 490, 0, 7]
    pairs["b_pos"] = [0, 20, 300, 590, 5, 0]
    pairs["a_len"] = [5, 30, 200, 10, 0, 3]
    pairs["b_len"] = [5, 40, 250, 10, 4, 0]
    f = oracle.edit_distance if fn == "edit" else oracle.dtw
    got = oracle.pairs_batch(f, a, b, pairs)
    for k, pr in enumerate(pairs):
        sa = a[pr["a_pos"]:pr["a_pos"] + pr["a_len"]]
        sb = b[pr["b_pos"]:pr["b_pos"] + pr["b_len"]]
        assert got[k] == f(sa, sb)
