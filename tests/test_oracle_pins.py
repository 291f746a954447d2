"""Pins for the CPU oracle: it is checked against things other than itself.

* enumeration of every alignment on tiny windows (unpruned extension and local
  alignment), with random non-symmetric scoring matrices so that a transposed
  operand, a wrong sign or a dropped term shows up;
* hand-derived closed forms (tests/golden/closed_forms.json);
* re-scoring of every emitted CIGAR by an independent scorer;
* invariance to the visiting order inside an anti-diagonal and to batch order;
* pruning can only lower the score; the left side equals the right side on
  reversed sequences.
"""
import json
import os

import numpy as np
import pytest

from gapped_smith_waterman_gb300 import workloads as W
from tests import refcheck as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")
CODE = {"A": 0, "C": 1, "G": 2, "T": 3}


def enc(s):
    return np.array([CODE[c] for c in s], np.uint8)


def cigar_str(runs):
    return "".join(f"{int(r) >> 4}{'MID'[int(r) & 15]}" for r in runs)


def test_golden_closed_forms(oracle_lib):
    cases = json.load(open(GOLDEN))["cases"]
    assert len(cases) >= 10
    for c in cases:
        t, q, ex = enc(c["target"]), enc(c["query"]), c["expect"]
        if c["mode"] == "local":
            got = oracle_lib.local_one(t, q, W.HOXD70, 400, 30)
            assert got == (ex["score"], ex["i_end"], ex["j_end"]), c["name"]
            continue
        s, i, j, live, _, runs = oracle_lib.extend_one(t, q, W.HOXD70, 400, 30, c["ydrop"])
        assert (s, i, j) == (ex["score"], ex["i_end"], ex["j_end"]), c["name"]
        assert cigar_str(runs) == ex["cigar"], c["name"]
        if "live_cells" in ex:
            assert live == ex["live_cells"], c["name"]


def _random_case(rng, max_len=6, alphabet_bias=True):
    m = int(rng.integers(0, max_len + 1))
    n = int(rng.integers(0, max_len + 1))
    t = rng.integers(0, 4, m).astype(np.uint8)
    if alphabet_bias and m and rng.random() < 0.6:
        # query related to the target so that long alignments win sometimes
        q = t.copy()
        for k in range(q.size):
            if rng.random() < 0.25:
                q[k] = rng.integers(0, 4)
        q = q[:n] if n <= q.size else np.concatenate([q, rng.integers(0, 4, n - q.size).astype(np.uint8)])
    else:
        q = rng.integers(0, 4, n).astype(np.uint8)
    return t, q


def _random_scoring(rng):
    sub = rng.integers(-60, 61, size=(4, 4)).astype(np.int32)
    sub[np.arange(4), np.arange(4)] = rng.integers(20, 101, 4)
    o = int(rng.integers(1, 80))
    e = int(rng.integers(1, 40))
    return sub, o, e


def _tie_scoring(rng):
    """Uniform match/mismatch with small gap costs: equal scores everywhere,
    so end-cell and traceback tie rules decide most cases."""
    mt = int(rng.integers(2, 6))
    sub = np.full((4, 4), -mt, np.int32)
    sub[np.arange(4), np.arange(4)] = mt
    return sub, int(rng.integers(1, 4)), int(rng.integers(1, 4))


def _scoring(rng, it):
    return (_random_scoring(rng), _tie_scoring(rng), (W.HOXD70, 400, 30))[it % 3]


@pytest.mark.parametrize("seed", range(6))
def test_bruteforce_extend_unpruned(oracle_lib, seed):
    rng = np.random.default_rng(1000 + seed)
    for it in range(40):
        t, q = _random_case(rng)
        sub, o, e = _scoring(rng, it)
        want = R.brute_extend(t, q, sub, o, e)
        for desc in (False, True):
            s, i, j, live, _, runs = oracle_lib.extend_one(t, q, sub, o, e, -1, descending=desc)
            assert (s, i, j) == want[:3], (t, q, sub, o, e)
            assert R.runs_to_ops(runs) == want[3], (t, q, sub, o, e)
            assert live == (len(t) + 1) * (len(q) + 1)


@pytest.mark.parametrize("seed", range(4))
def test_bruteforce_local(oracle_lib, seed):
    rng = np.random.default_rng(2000 + seed)
    for it in range(25):
        t, q = _random_case(rng, max_len=5)
        sub, o, e = _scoring(rng, it)
        assert oracle_lib.local_one(t, q, sub, o, e) == R.brute_local(t, q, sub, o, e), (t, q, sub, o, e)


def test_bruteforce_local_vs_textbook_sizes(oracle_lib):
    # one-sided extension and local alignment agree when the best local
    # alignment is anchored at the origin: identical prefixes, mismatching tails
    rng = np.random.default_rng(7)
    for _ in range(20):
        x = rng.integers(0, 4, int(rng.integers(1, 40))).astype(np.uint8)
        tail_t = np.zeros(10, np.uint8)           # A ...
        tail_q = np.ones(10, np.uint8)            # ... against C
        t = np.concatenate([x, tail_t])
        q = np.concatenate([x, tail_q])
        loc = oracle_lib.local_one(t, q, W.HOXD70, 400, 30)
        ext = oracle_lib.extend_one(t, q, W.HOXD70, 400, 30, -1)
        assert loc == ext[:3] == (int(W.HOXD70[x, x].sum()), x.size, x.size)


def test_identical_closed_form(oracle_lib):
    rng = np.random.default_rng(11)
    for L in list(range(1, 30)) + [64, 99, 100]:
        x = rng.integers(0, 4, L).astype(np.uint8)
        want = int(W.HOXD70[x, x].sum())
        for yd in (9400, -1):
            s, i, j, _, _, runs = oracle_lib.extend_one(x, x, W.HOXD70, 400, 30, yd)
            assert (s, i, j) == (want, L, L)
            assert cigar_str(runs) == f"{L}M"


@pytest.mark.parametrize("k", [1, 2, 5, 17, 40])
def test_single_gap_closed_form(oracle_lib, k):
    rng = np.random.default_rng(100 + k)
    # P and R over {C,G,T}; the gap block is all A, so it never matches
    P = rng.integers(1, 4, 30).astype(np.uint8)
    Rr = rng.integers(1, 4, 60).astype(np.uint8)
    G = np.zeros(k, np.uint8)
    sP = int(W.HOXD70[P, P].sum())
    sR = int(W.HOXD70[Rr, Rr].sum())
    want = sP + sR - (400 + 30 * k)
    # deletion (target has the extra block)
    s, i, j, _, _, runs = oracle_lib.extend_one(np.concatenate([P, G, Rr]), np.concatenate([P, Rr]),
                                                W.HOXD70, 400, 30, 9400)
    assert (s, i, j) == (want, 90 + k, 90) and cigar_str(runs) == f"30M{k}D60M"
    # insertion (query has the extra block)
    s, i, j, _, _, runs = oracle_lib.extend_one(np.concatenate([P, Rr]), np.concatenate([P, G, Rr]),
                                                W.HOXD70, 400, 30, 9400)
    assert (s, i, j) == (want, 90, 90 + k) and cigar_str(runs) == f"30M{k}I60M"


@pytest.mark.parametrize("k", [3, 10, 50])
def test_gap_threshold_is_strict(oracle_lib, k):
    rng = np.random.default_rng(200 + k)
    P = rng.integers(1, 4, 20).astype(np.uint8)
    Rr = rng.integers(1, 4, 120).astype(np.uint8)
    t = np.concatenate([P, np.zeros(k, np.uint8), Rr])
    q = np.concatenate([P, Rr])
    sP = int(W.HOXD70[P, P].sum())
    sR = int(W.HOXD70[Rr, Rr].sum())
    cost = 400 + 30 * k
    assert sR > cost
    s, i, j, _, _, _ = oracle_lib.extend_one(t, q, W.HOXD70, 400, 30, cost)
    assert (s, i, j) == (sP + sR - cost, 140 + k, 140)
    s, i, j, _, _, runs = oracle_lib.extend_one(t, q, W.HOXD70, 400, 30, cost - 1)
    assert (s, i, j) == (sP, 20, 20) and cigar_str(runs) == "20M"


def test_diagonal_only_live_count(oracle_lib):
    # ydrop = open + extend - 1: only the diagonal survives; pins that the
    # threshold includes the anti-diagonal just completed and that the sweep
    # goes on past an anti-diagonal without live cells
    rng = np.random.default_rng(5)
    for L in (1, 2, 7, 33):
        x = rng.integers(0, 4, L).astype(np.uint8)
        s, i, j, live, _, _ = oracle_lib.extend_one(x, x, W.HOXD70, 400, 30, 429)
        assert (s, i, j, live) == (int(W.HOXD70[x, x].sum()), L, L, L + 1)


def test_cigar_rescores_on_short_windows(oracle_lib):
    w = W.make_cfg1(n_pairs=400)
    res, cig, off = oracle_lib.extend_batch(w, nthreads=4)
    for k in range(len(w.seeds)):
        r = res[2 * k]
        runs = cig[off[2 * k]:off[2 * k] + r["n_cigar"]]
        t = W.window_bases(w.target, w.seeds["t_pos"][k], W.SIDE_RIGHT, w.max_len)
        q = W.window_bases(w.query, w.seeds["q_pos"][k], W.SIDE_RIGHT, w.max_len)
        s, i, j = R.rescore_cigar(runs, t, q, W.HOXD70, 400, 30)
        assert (s, i, j) == (r["score"], r["i_end"], r["j_end"])
        # runs are maximal (adjacent runs differ)
        ops = [int(x) & 15 for x in runs]
        assert all(a != b for a, b in zip(ops, ops[1:]))
    assert res["status"].max() == 0
    assert res["score"][1::2].max() == 0            # left sides not requested


def test_cigar_rescores_small_ydrop(oracle_lib):
    rng = np.random.default_rng(9)
    for _ in range(200):
        t, q = _random_case(rng, max_len=40)
        yd = int(rng.integers(0, 1500))
        s, i, j, _, _, runs = oracle_lib.extend_one(t, q, W.HOXD70, 400, 30, yd)
        assert R.rescore_cigar(runs, t, q, W.HOXD70, 400, 30) == (s, i, j)


def test_order_invariance(oracle_lib):
    w = W.make_cfg1(n_pairs=300)
    a = oracle_lib.extend_batch(w, nthreads=4, descending=False)
    b = oracle_lib.extend_batch(w, nthreads=4, descending=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # small ydrop makes pruning decisions dense
    for yd in (0, 100, 429, 430, 700):
        a = oracle_lib.extend_batch(w, nthreads=4, ydrop=yd)
        b = oracle_lib.extend_batch(w, nthreads=4, ydrop=yd, descending=True)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # batch order
    perm = np.random.default_rng(3).permutation(len(w.seeds))
    a = oracle_lib.extend_batch(w, nthreads=4)
    b = oracle_lib.extend_batch(w, seeds=w.seeds[perm], nthreads=3)
    for k, p in enumerate(perm):
        assert a[0][2 * p] == b[0][2 * k]


def test_pruning_only_lowers_score(oracle_lib):
    rng = np.random.default_rng(13)
    for _ in range(150):
        t, q = _random_case(rng, max_len=60)
        s_inf = oracle_lib.extend_one(t, q, W.HOXD70, 400, 30, -1)
        for yd in (0, 300, 1000, 9400):
            s = oracle_lib.extend_one(t, q, W.HOXD70, 400, 30, yd)
            assert s[0] <= s_inf[0]
            assert s[3] <= s_inf[3]          # live cells


def test_huge_ydrop_equals_unpruned(oracle_lib):
    rng = np.random.default_rng(17)
    for _ in range(50):
        t, q = _random_case(rng, max_len=50)
        a = oracle_lib.extend_one(t, q, W.HOXD70, 400, 30, -1)
        b = oracle_lib.extend_one(t, q, W.HOXD70, 400, 30, 1 << 28)
        assert a[:5] == b[:5] and np.array_equal(a[5], b[5])


def test_left_side_is_right_side_on_reversed_sequences(oracle_lib):
    rng = np.random.default_rng(21)
    tseq = rng.integers(0, 4, 3000).astype(np.uint8)
    qseq = W.mutate(rng, tseq, 0.1, 0.01, 2.0)
    n = 60
    seeds = np.zeros(n, W.SEED_DTYPE)
    seeds["t_pos"] = rng.integers(0, tseq.size + 1, n)
    seeds["q_pos"] = np.minimum(seeds["t_pos"] + rng.integers(-5, 6, n), qseq.size).clip(0)
    seeds["side"] = W.SIDE_BOTH
    w = W.Workload("t", tseq, qseq, seeds, W.HOXD70, 400, 30, 9400, 500, 0)
    res, cig, off = oracle_lib.extend_batch(w, nthreads=2)
    rs = seeds.copy()
    rs["t_pos"] = tseq.size - seeds["t_pos"]
    rs["q_pos"] = qseq.size - seeds["q_pos"]
    rs["side"] = W.SIDE_RIGHT
    wr = W.Workload("r", tseq[::-1].copy(), qseq[::-1].copy(), rs, W.HOXD70, 400, 30, 9400, 500, 0)
    rres, rcig, roff = oracle_lib.extend_batch(wr, nthreads=2)
    for k in range(n):
        a, b = res[2 * k + 1], rres[2 * k]
        assert (a["score"], a["i_end"], a["j_end"], a["live_cells"]) == \
               (b["score"], b["i_end"], b["j_end"], b["live_cells"])
        assert np.array_equal(cig[off[2 * k + 1]:off[2 * k + 1] + a["n_cigar"]],
                              rcig[roff[2 * k]:roff[2 * k] + b["n_cigar"]])


def test_planted_mistakes_are_caught():
    """A transposed matrix or an off-by-one gap cost in a re-implementation
    would be caught by the brute force: check the brute force itself separates
    them on the pinned inputs."""
    rng = np.random.default_rng(1)
    sub, o, e = _random_scoring(rng)
    assert not np.array_equal(sub, sub.T)
    seen_t = seen_gap = False
    for _ in range(200):
        t, q = _random_case(rng)
        a = R.brute_extend(t, q, sub, o, e)
        if a[:3] != R.brute_extend(t, q, sub.T.copy(), o, e)[:3]:
            seen_t = True
        if a[:3] != R.brute_extend(t, q, sub, o - e, e)[:3]:
            seen_gap = True
        if seen_t and seen_gap:
            break
    assert seen_t and seen_gap


def test_end_cell_tie_on_one_antidiagonal(oracle_lib):
    """t = AC, q = CA with match 5, mismatch -5, gap open 1, extend 1.
    (1,2) = I(0,1) then A/A: -2 + 5 = 3; (2,1) = D(1,0) then C/C: -2 + 5 = 3;
    both lie on anti-diagonal 3 and nothing scores more ((2,2) <= 1), so the
    earliest cell by (d, i) is (1,2).  Local mode: the same two cells score 5
    (the zero floor replaces the gap) on anti-diagonal 3, and (1,2) wins."""
    sub = np.full((4, 4), -5, np.int32)
    sub[np.arange(4), np.arange(4)] = 5
    t, q = enc("AC"), enc("CA")
    s, i, j, _, _, runs = oracle_lib.extend_one(t, q, sub, 1, 1, -1)
    assert (s, i, j) == (3, 1, 2) and cigar_str(runs) == "1I1M"
    s, i, j, _, _, runs = oracle_lib.extend_one(q, t, sub, 1, 1, -1)
    assert (s, i, j) == (3, 1, 2) and cigar_str(runs) == "1I1M"
    assert oracle_lib.local_one(t, q, sub, 1, 1) == (5, 1, 2)
    # mirrored: t = CA, q = AC -> cells (1,2) and (2,1) again
    s, i, j, _, _, _ = oracle_lib.extend_one(enc("GAC"), enc("GCA"), sub, 1, 1, -1)
    assert (s, i, j) == (8, 2, 3)


# ---- two-sided combination (FastZ, section 3.1.2: LASTZ joins the two sides) ----

def _pair_workload(t, q, seeds, max_len=200):
    return W.Workload("pair", np.asarray(t, np.uint8), np.asarray(q, np.uint8), seeds,
                      np.asarray(W.HOXD70, np.int32), 400, 30, 9400, max_len, W.MODE_EXTEND)


def _cigar_str(runs):
    return "".join(f"{int(r) >> 4}{'MID'[int(r) & 15]}" for r in runs)


def test_combine_identical_region_is_one_match_run(oracle_lib):
    """A seed inside an identical region: the two sides meet at the anchor, so
    the combined alignment is the whole region, one M run, scoring the sum of
    the diagonal terms."""
    import oracle
    rng = np.random.default_rng(11)
    t = rng.integers(0, 4, 40).astype(np.uint8)
    sub = np.asarray(W.HOXD70, np.int64).reshape(4, 4)
    seeds = np.zeros(1, W.SEED_DTYPE)
    seeds["t_pos"], seeds["q_pos"], seeds["side"] = 15, 15, W.SIDE_BOTH
    w = _pair_workload(t, t.copy(), seeds)
    res, cig, off = oracle.extend_batch(w)
    (score, ts, qs, te, qe, runs), = oracle.combine(seeds, res, cig, off)
    assert score == int(sum(sub[a, a] for a in t))
    assert (ts, qs, te, qe) == (0, 0, 40, 40)
    assert _cigar_str(runs) == "40M"


def test_combine_gap_on_the_left_side(oracle_lib):
    """A 3-base deletion 10 bases left of the anchor: the left side carries it,
    the right side is all matches, and the runs join as 10M 3D (10+20)M."""
    import oracle
    rng = np.random.default_rng(12)
    q = rng.integers(0, 4, 40).astype(np.uint8)
    t = np.concatenate([q[:10], rng.integers(0, 4, 3).astype(np.uint8), q[10:]])   # 3 extra target bases
    sub = np.asarray(W.HOXD70, np.int64).reshape(4, 4)
    seeds = np.zeros(1, W.SEED_DTYPE)
    seeds["t_pos"], seeds["q_pos"], seeds["side"] = 23, 20, W.SIDE_BOTH   # anchor after 20 query bases
    w = _pair_workload(t, q, seeds)
    res, cig, off = oracle.extend_batch(w)
    (score, ts, qs, te, qe, runs), = oracle.combine(seeds, res, cig, off)
    assert _cigar_str(runs) == "10M3D30M"
    assert (ts, qs, te, qe) == (0, 0, 43, 40)
    assert score == int(sum(sub[a, a] for a in q)) - (400 + 3 * 30)


def test_combine_one_side_only(oracle_lib):
    import oracle
    rng = np.random.default_rng(13)
    t = rng.integers(0, 4, 30).astype(np.uint8)
    seeds = np.zeros(2, W.SEED_DTYPE)
    seeds["t_pos"], seeds["q_pos"] = 10, 10
    seeds["side"] = [W.SIDE_RIGHT, W.SIDE_LEFT]
    w = _pair_workload(t, t.copy(), seeds)
    res, cig, off = oracle.extend_batch(w)
    right, left = oracle.combine(seeds, res, cig, off)
    assert (right[0], right[1], right[3], _cigar_str(right[5])) == (int(res["score"][0]), 10, 30, "20M")
    assert (left[0], left[1], left[3], _cigar_str(left[5])) == (int(res["score"][3]), 0, 10, "10M")
