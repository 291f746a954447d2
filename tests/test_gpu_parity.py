"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Scores, end cells, CIGARs and flags must be bit-exact (integer work).  Every
workload, full-size ones included, is compared on every extension: directly
against an oracle run in the test, or (the 2,000,000 extensions of the
chromosome batch, hours of oracle time) against stored digests of an oracle
run over the same seeded inputs.
"""
import json
import os

import numpy as np
import pytest

from gapped_smith_waterman_gb300 import workloads as W
from tests import gpu_common as G
from tests import refcheck as R

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from gapped_smith_waterman_gb300 import build
    build.build()
    import oracle
    oracle.lib()


def _one_pair_workload(t, q, sub=W.HOXD70, o=400, e=30, ydrop=9400, mode=W.MODE_EXTEND, side=W.SIDE_RIGHT):
    t = np.asarray(t, np.uint8)
    q = np.asarray(q, np.uint8)
    seeds = np.zeros(1, W.SEED_DTYPE)
    seeds["side"] = side
    if side == W.SIDE_LEFT:
        seeds["t_pos"] = t.size
        seeds["q_pos"] = q.size
        t, q = t[::-1].copy(), q[::-1].copy()
    ml = max(1, t.size, q.size)
    return W.Workload("pair", t, q, seeds, np.asarray(sub, np.int32), o, e, ydrop, ml, mode)


def _batch_from_pairs(pairs, sub=W.HOXD70, o=400, e=30, ydrop=9400, mode=W.MODE_EXTEND):
    """Pairs laid end to end; seed k anchors at the start of pair k; max_len
    = the longest window, each pair padded so windows never overlap."""
    ml = max(1, max(max(len(t), len(q)) for t, q in pairs))
    T = np.zeros(len(pairs) * ml, np.uint8)          # padding A in the target ...
    Q = np.ones(len(pairs) * ml, np.uint8)           # ... against C in the query: windows stop at pair ends
    seeds = np.zeros(len(pairs), W.SEED_DTYPE)
    tl = []
    for k, (t, q) in enumerate(pairs):
        T[k * ml:k * ml + len(t)] = t
        Q[k * ml:k * ml + len(q)] = q
        seeds[k]["t_pos"] = k * ml
        seeds[k]["q_pos"] = k * ml
        tl.append((len(t), len(q)))
    seeds["side"] = W.SIDE_RIGHT
    return W.Workload("pairs", T, Q, seeds, np.asarray(sub, np.int32), o, e, ydrop, ml, mode), tl


def _check(w, seeds=None, label="", check_cigar=True):
    gres, gcig, st = G.gpu_run(w, seeds)
    ores, ocig, ooff = G.oracle_run(w, seeds)
    G.compare(w, seeds, gres, gcig, ores, ocig, ooff, check_cigar=check_cigar, label=label)
    return gres, gcig, st, ores


def test_golden_closed_forms_gpu():
    cases = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))["cases"]
    code = {"A": 0, "C": 1, "G": 2, "T": 3}
    for c in cases:
        t = np.array([code[x] for x in c["target"]], np.uint8)
        q = np.array([code[x] for x in c["query"]], np.uint8)
        mode = W.MODE_LOCAL if c["mode"] == "local" else W.MODE_EXTEND
        yd = c.get("ydrop", W.YDROP_INF)
        w = _one_pair_workload(t, q, ydrop=yd, mode=mode)
        gres, gcig, st = G.gpu_run(w)
        ex = c["expect"]
        g = gres[0]
        assert (g["score"], g["t_end"], g["q_end"]) == (ex["score"], ex["i_end"], ex["j_end"]), c["name"]
        if mode == W.MODE_EXTEND:
            runs = gcig[g["cigar_off"]:g["cigar_off"] + g["cigar_len"]]
            assert "".join(f"{int(r) >> 4}{'MID'[int(r) & 15]}" for r in runs) == ex["cigar"], c["name"]
            if "live_cells" in ex:
                assert st.live_cells == ex["live_cells"], c["name"]


def test_cfg1_full():
    w = G.workload(1)
    gres, gcig, st, ores = _check(w, label="short-256bp")
    assert st.live_cells == int(ores["live_cells"].sum())
    assert st.extensions == len(w.seeds)
    assert st.eager + sum(st.bin) + st.traced == st.extensions


def test_cfg2_subset_all_fields():
    w = G.workload(2)
    idx = np.arange(4000)
    gres, gcig, st, ores = _check(w, w.seeds[idx], label="skewed-6kbp[:4000]")
    assert st.live_cells == int(ores["live_cells"].sum())


def test_cfg2_every_extension():
    """All 100,000 extensions of the 6 kbp batch in one launch, every field
    against the oracle, and the batch's live-cell total."""
    w = G.workload(2)
    gres, gcig, st, ores = _check(w, label="skewed-6kbp, every extension")
    assert st.live_cells == int(ores["live_cells"].sum())
    assert st.extensions == len(w.seeds)
    # CIGARs re-score to their records (an independent scorer, not the oracle)
    for k in G.sample_seeds(w, 3000, seed=5):
        g = gres[2 * k]
        runs = gcig[g["cigar_off"]:g["cigar_off"] + g["cigar_len"]]
        t = W.window_bases(w.target, w.seeds["t_pos"][k], W.SIDE_RIGHT, w.max_len)
        q = W.window_bases(w.query, w.seeds["q_pos"][k], W.SIDE_RIGHT, w.max_len)
        assert R.rescore_cigar(runs, t, q, w.sub, w.gap_open, w.gap_extend) == (g["score"], g["t_end"], g["q_end"])


def _cfg3_host_run(w):
    """The whole chromosome batch through the device entry, then again
    through the host entry (packed runs); both must agree."""
    from gapped_smith_waterman_gb300 import fz
    ext = fz.Extender.for_workload(w)
    try:
        d_t, d_q, d_s = ext.upload(W.pack2(w.target), W.pack2(w.query), w.seeds)
        d_out = ext.alloc_out(len(w.seeds))
        ext.run(d_t, w.target.size, d_q, w.query.size, d_s, len(w.seeds), d_out)
        st = ext.stats()
        dres = np.frombuffer(d_out[:2 * len(w.seeds) * fz.RESULT_DTYPE.itemsize].cpu().numpy().tobytes(),
                             dtype=fz.RESULT_DTYPE)
        used = int(dres["cigar_len"].astype(np.int64).sum())
        del d_t, d_q, d_s, d_out
        hres, packed = ext.extend_workload_host(w, cigar_cap=used + 16)
        st2 = ext.stats()
    finally:
        ext.close()
    for f in ("score", "t_end", "q_end", "cigar_len", "flags"):
        assert np.array_equal(dres[f], hres[f]), f
    assert packed.size == used and st.live_cells == st2.live_cells
    return hres, packed, st


def test_cfg3_every_extension():
    """All 2,000,000 one-sided extensions of the chromosome batch against the
    oracle: per chunk of 4,096 seeds, the digest of score, end cell and CIGAR
    of every extension equals the one stored by tests/golden/make_oracle_digests.py
    (a run of the CPU oracle over the same seeded inputs), and the live-cell
    total equals the oracle's.  A differing chunk is re-run on the oracle here
    to name the first differing extension.  If the generated inputs differ from
    the ones the digests were made from (another numpy's random streams), the
    test falls back to 50,000 sampled seeds compared field by field."""
    from tests import digest as D
    w = G.workload(3)
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_digest_cfg3.json")
    doc = json.load(open(path)) if os.path.exists(path) else None
    usable = (doc is not None and doc["input_sha256"] == D.input_sha256(w) and
              all(c is not None for c in doc["chunks"]))
    if not usable:
        gres, gcig, st = G.gpu_run(w)
        idx = G.sample_seeds(w, 50_000, seed=3)
        ores, ocig, ooff = G.oracle_run(w, w.seeds[idx])
        xs = np.stack([2 * idx, 2 * idx + 1], 1).reshape(-1)
        G.compare(G.sub_workload(w, idx), None, gres[xs], gcig, ores, ocig, ooff, label="chrom-50Mbp sampled")
        assert st.extensions == 2 * len(w.seeds)
        pytest.skip("stored digests do not match these inputs: compared 50,000 sampled seeds instead")
    hres, packed, st = _cfg3_host_run(w)
    assert st.extensions == 2 * len(w.seeds)
    assert st.live_cells == sum(doc["live_cells"])
    cs = doc["chunk_seeds"]
    bad = []
    for c, want in enumerate(doc["chunks"]):
        x0, x1 = 2 * c * cs, 2 * min(len(w.seeds), (c + 1) * cs)
        if D.chunk_digest(*D.packed_chunk(hres, packed, x0, x1)) != want:
            bad.append(c)
    if bad:
        c = bad[0]
        idx = np.arange(c * cs, min(len(w.seeds), (c + 1) * cs))
        ores, ocig, ooff = G.oracle_run(w, w.seeds[idx])
        sub = hres[2 * idx[0]:2 * (idx[-1] + 1)]
        G.compare(G.sub_workload(w, idx), None, sub, packed, ores, ocig, ooff, label=f"chrom-50Mbp chunk {c}")
        pytest.fail(f"{len(bad)} chunks differ from the stored oracle digests (first {c}), "
                    "but the oracle re-run of the first agrees: stale digests?")


def test_cfg4_every_extension():
    """All 2,000 long extensions (60 kbp windows): the executor's big bins,
    many segments per extension and the longest traceback walks."""
    w = G.workload(4)
    gres, gcig, st, ores = _check(w, label="long-60kbp, every extension")
    assert st.live_cells == int(ores["live_cells"].sum())


def test_cfg5_every_pair():
    """All 65,536 local fills of 2,048 x 2,048."""
    w = G.workload(5)
    gres, gcig, st, ores = _check(w, label="local-2048, every pair", check_cigar=False)
    assert st.live_cells == len(w.seeds) * 2048 * 2048 == int(ores["live_cells"].sum())


def test_edge_cases():
    rng = np.random.default_rng(42)
    code = lambda s: np.array(["ACGT".index(c) for c in s], np.uint8)  # noqa: E731
    x = rng.integers(0, 4, 200).astype(np.uint8)
    pairs = [
        (np.zeros(0, np.uint8), np.zeros(0, np.uint8)),          # empty windows
        (code("A"), code("A")),                                   # window of 1
        (code("A"), np.zeros(0, np.uint8)),
        (np.zeros(0, np.uint8), code("ACGT")),
        (np.zeros(30, np.uint8), np.ones(30, np.uint8)),         # all mismatch
        (x, x),                                                   # identical
        (x[:16], x[:16]),                                         # ends exactly at (16,16)
        (x[:17], x[:16]),
        (x[:16], x[:17]),
        (np.concatenate([x[:17], code("AA")]), np.concatenate([x[:16], code("CC")])),
        (np.concatenate([x[:80], np.zeros(60, np.uint8), x[80:]]), x),   # single long gap
        (x[:100], np.concatenate([x[:50], x[60:100]])),
    ]
    # bin edges: identical prefixes ending at 512 and 513
    for L in (511, 512, 513):
        y = rng.integers(0, 4, L).astype(np.uint8)
        pairs.append((np.concatenate([y, np.zeros(40, np.uint8)]), np.concatenate([y, np.ones(40, np.uint8)])))
    w, _ = _batch_from_pairs(pairs)
    _check(w, label="edge cases")
    for yd in (0, 1, 429, 430, 5000, W.YDROP_INF):
        w2 = W.Workload(w.name, w.target, w.query, w.seeds, w.sub, w.gap_open, w.gap_extend, yd, w.max_len, w.mode)
        _check(w2, label=f"edge cases ydrop={yd}")


def test_edge_cases_inspector_and_executor(monkeypatch):
    """The edge cases with the traced sweep off: windows this short otherwise all
    take it, so the plain inspector, bins, executor and walk run here."""
    monkeypatch.setenv("FZ_TRACED", "0")
    test_edge_cases()
    test_left_and_both_sides_and_sequence_ends()


def test_left_and_both_sides_and_sequence_ends():
    rng = np.random.default_rng(7)
    t = rng.integers(0, 4, 5000).astype(np.uint8)
    q = W.mutate(rng, t, 0.08, 0.01, 2.0)
    n = 300
    seeds = np.zeros(n, W.SEED_DTYPE)
    seeds["t_pos"] = rng.integers(0, t.size + 1, n)
    seeds["q_pos"] = np.clip(seeds["t_pos"].astype(np.int64) + rng.integers(-3, 4, n), 0, q.size)
    seeds["side"] = rng.integers(1, 4, n)
    seeds[0]["t_pos"], seeds[0]["q_pos"], seeds[0]["side"] = 0, 0, 3
    seeds[1]["t_pos"], seeds[1]["q_pos"], seeds[1]["side"] = t.size, q.size, 3
    seeds[2]["t_pos"], seeds[2]["q_pos"], seeds[2]["side"] = t.size, 0, 3
    w = W.Workload("sides", t, q, seeds, W.HOXD70.copy(), 400, 30, 9400, 700, W.MODE_EXTEND)
    _check(w, label="sides")


@pytest.mark.parametrize("seed", range(4))
def test_fuzz_small_random_parameters(seed, monkeypatch):
    # windows this short take the traced sweep; seeds 2 and 3 turn it off so
    # that the plain inspector and the executor see the same kind of batches
    if seed >= 2:
        monkeypatch.setenv("FZ_TRACED", "0")
    rng = np.random.default_rng(300 + seed)
    for it in range(6):
        sub = rng.integers(-120, 121, size=(4, 4)).astype(np.int32)
        sub[np.arange(4), np.arange(4)] = rng.integers(20, 128, 4)
        o = int(rng.integers(0, 600))
        e = int(rng.integers(1, 60))
        yd = int(rng.choice([0, 50, 300, 800, 2000, 9400, W.YDROP_INF]))
        pairs = []
        for _ in range(150):
            m = int(rng.integers(0, 300))
            t = rng.integers(0, 4, m).astype(np.uint8)
            q = W.mutate(rng, t[:int(rng.integers(0, m + 1))], rng.uniform(0, 0.3), rng.uniform(0, 0.05), 2.0)
            q = np.concatenate([q, rng.integers(0, 4, int(rng.integers(0, 60))).astype(np.uint8)])
            pairs.append((t, q))
        w, _ = _batch_from_pairs(pairs, sub=sub, o=o, e=e, ydrop=yd)
        _check(w, label=f"fuzz seed={seed} it={it} o={o} e={e} ydrop={yd}")


def test_local_fuzz():
    rng = np.random.default_rng(77)
    for it in range(4):
        sub = rng.integers(-100, 101, size=(4, 4)).astype(np.int32)
        sub[np.arange(4), np.arange(4)] = rng.integers(20, 128, 4)
        pairs = []
        for _ in range(60):
            m = int(rng.integers(0, 1500))
            t = rng.integers(0, 4, m).astype(np.uint8)
            q = W.mutate(rng, t, 0.2, 0.02, 2.0) if rng.random() < 0.5 else rng.integers(0, 4, int(rng.integers(0, 2500))).astype(np.uint8)
            pairs.append((t, q))
        w, _ = _batch_from_pairs(pairs, sub=sub, o=int(rng.integers(0, 500)), e=int(rng.integers(1, 50)),
                                 ydrop=W.YDROP_INF, mode=W.MODE_LOCAL)
        _check(w, label=f"local fuzz {it}", check_cigar=False)


def test_wide_band_path():
    # ydrop far above the register window's reach: gaps of thousands stay live
    rng = np.random.default_rng(8)
    pairs = []
    for _ in range(24):
        t = rng.integers(0, 4, 1500).astype(np.uint8)
        q = W.mutate(rng, t, 0.1, 0.02, 3.0)
        pairs.append((t, q))
    w, _ = _batch_from_pairs(pairs, ydrop=40000)
    gres, gcig, st, ores = _check(w, label="wide band")
    assert st.wide > 0


def test_wide_band_beyond_the_ring():
    """Bands wider than the wide path's 2,048-row shared-memory ring (no
    y-drop, windows of 2,300 to 2,700 bases, homologous and unrelated pairs):
    the block moves its anti-diagonals to the global scratch mid-sweep, in the
    inspector and in the executor; records and CIGARs equal the oracle's."""
    rng = np.random.default_rng(12)
    pairs = []
    for L in (2300, 2500, 2700):
        t = rng.integers(0, 4, L).astype(np.uint8)
        pairs.append((t, W.mutate(rng, t, 0.1, 0.02, 3.0)))
        pairs.append((t, rng.integers(0, 4, L).astype(np.uint8)))
    w, _ = _batch_from_pairs(pairs, ydrop=W.YDROP_INF)
    gres, gcig, st, ores = _check(w, label="wide band beyond the ring")
    assert st.wide == len(pairs)


def test_wide_band_both_sides():
    """Two-sided anchors in the middle of long homologous pairs at y-drop
    40,000: both extensions of every seed take the wide path, the left one
    reading its windows backwards (the staged bases in reverse order), with
    windows short enough to be staged and, in a second batch, too long."""
    rng = np.random.default_rng(14)
    for L, mid in ((3000, 1400), (9000, 4300)):
        T, Q, seeds = [], [], np.zeros(3, W.SEED_DTYPE)
        for k in range(3):
            t = rng.integers(0, 4, L).astype(np.uint8)
            q = W.mutate(rng, t, 0.1, 0.02, 3.0)[:L]
            q = np.concatenate([q, rng.integers(0, 4, L - q.size).astype(np.uint8)])
            seeds[k]["t_pos"] = k * L + mid
            seeds[k]["q_pos"] = k * L + mid + int(rng.integers(-3, 4))
            T.append(t)
            Q.append(q)
        seeds["side"] = W.SIDE_BOTH
        w = W.Workload("both", np.concatenate(T), np.concatenate(Q), seeds, W.HOXD70.copy(), 400, 30, 40000,
                       L // 2 - 100 if L < 5000 else L // 2, W.MODE_EXTEND)
        gres, gcig, st, ores = _check(w, label=f"wide band, both sides, {L} bp pairs")
        assert st.wide >= 4


def test_wide_band_long_windows():
    """Windows longer than the wide path stages in shared memory (4,080
    bases): it reads the bases from global memory instead; records and
    CIGARs equal the oracle's."""
    rng = np.random.default_rng(13)
    pairs = []
    for L in (4200, 4400):
        t = rng.integers(0, 4, L).astype(np.uint8)
        pairs.append((t, W.mutate(rng, t, 0.1, 0.02, 3.0)))
    w, _ = _batch_from_pairs(pairs, ydrop=40000)
    assert w.max_len > 4080
    gres, gcig, st, ores = _check(w, label="wide band, long windows")
    assert st.wide == len(pairs)


def test_wide_band_fuzz():
    """The wide-band sweep on random non-symmetric scorings (a transposed
    substitution lookup fails here) with no y-drop: every band outgrows the
    512-row tier, some also the 2,048-row ring; then a matrix outside the
    byte range, which sends every extension to the wide path from the start."""
    rng = np.random.default_rng(78)
    for it in range(3):
        sub = rng.integers(-120, 121, size=(4, 4)).astype(np.int32)
        sub[np.arange(4), np.arange(4)] = rng.integers(40, 128, 4)
        pairs = []
        for _ in range(10):
            L = int(rng.integers(600, 2300))
            t = rng.integers(0, 4, L).astype(np.uint8)
            q = W.mutate(rng, t, 0.15, 0.03, 3.0) if rng.random() < 0.7 else rng.integers(0, 4, L).astype(np.uint8)
            pairs.append((t, q))
        w, _ = _batch_from_pairs(pairs, sub=sub, o=int(rng.integers(50, 500)), e=int(rng.integers(5, 60)),
                                 ydrop=W.YDROP_INF)
        gres, gcig, st, ores = _check(w, label=f"wide fuzz {it}")
        assert st.wide == len(pairs)
    sub = rng.integers(-300, 301, size=(4, 4)).astype(np.int32)
    sub[np.arange(4), np.arange(4)] = rng.integers(150, 300, 4)
    pairs = [(rng.integers(0, 4, int(rng.integers(1, 400))).astype(np.uint8),) * 2 for _ in range(12)]
    pairs = [(t, W.mutate(rng, t, 0.1, 0.02, 2.0)) for (t, _) in pairs]
    w, _ = _batch_from_pairs(pairs, sub=sub, o=900, e=70, ydrop=20000)
    gres, gcig, st, ores = _check(w, label="wide fuzz, matrix outside the byte range")
    assert st.wide == 2 * len(pairs)     # every extension slot, both sides of each seed


def test_matrix_outside_byte_range_uses_general_path():
    rng = np.random.default_rng(9)
    sub = (W.HOXD70 * 3).astype(np.int32)          # entries beyond [-128, 127]
    pairs = [(rng.integers(0, 4, 200).astype(np.uint8),) * 2 for _ in range(10)]
    pairs += [(rng.integers(0, 4, 150).astype(np.uint8), rng.integers(0, 4, 170).astype(np.uint8)) for _ in range(10)]
    w, _ = _batch_from_pairs(pairs, sub=sub, o=1200, e=90, ydrop=28200)
    _check(w, label="x3 matrix")


def _runs_of(res, cig):
    return [cig[o:o + n].tolist() for o, n in zip(res["cigar_off"].astype(np.int64), res["cigar_len"].astype(np.int64))]


def test_host_entry_matches_device_entry():
    """Same records and CIGARs; the host copy packs the runs in extension order."""
    w = G.workload(1)
    a, acig, _ = G.gpu_run(w)
    b, bcig, _ = G.gpu_run(w, host=True)
    for f in ("score", "t_end", "q_end", "cigar_len", "flags"):
        assert np.array_equal(a[f], b[f]), f
    assert _runs_of(a, acig) == _runs_of(b, bcig)
    packed = np.concatenate([[0], np.cumsum(b["cigar_len"].astype(np.int64))[:-1]])
    assert np.array_equal(b["cigar_off"].astype(np.int64), packed)
    assert bcig.size == int(b["cigar_len"].sum())


def test_checkpoint_settings_give_identical_results(monkeypatch):
    """Window checkpoints change only where sweeps resume (the 512-row retry,
    executor segments), never a result: a checkpoint every 32 anti-diagonals
    (many segments per executor extension), none at all, and a pool that runs
    out part-way all give the oracle's records."""
    w = G.workload(2)
    idx = np.arange(3000)
    ores, ocig, ooff = G.oracle_run(w, w.seeds[idx])
    runs = {}
    for label, env in (("every32", {"FZ_CKPT_EVERY": "32"}), ("none", {"FZ_CKPT_SLOTS": "0"}),
                       ("pool300", {"FZ_CKPT_SLOTS": "300", "FZ_CKPT_EVERY": "32"})):
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        gres, gcig, st = G.gpu_run(w, w.seeds[idx])
        for k in env:
            monkeypatch.delenv(k)
        G.compare(w, w.seeds[idx], gres, gcig, ores, ocig, ooff, label=f"checkpoints {label}")
        assert st.live_cells == int(ores["live_cells"].sum()), label
        runs[label] = st
    # segments tile each replay (0, d*] exactly: the replayed rows do not depend on them
    assert runs["every32"].exec_cells == runs["none"].exec_cells == runs["pool300"].exec_cells


def test_checkpoints_long_alignments(monkeypatch):
    """Long alignments (60 kbp windows): many segments per extension."""
    monkeypatch.setenv("FZ_CKPT_EVERY", "64")
    w = G.workload(4)
    idx = G.sample_seeds(w, 12, seed=11)
    _check(w, w.seeds[idx], label="long-60kbp, checkpoint every 64")


def test_pair_sweep_equals_32bit_sweep(monkeypatch):
    """The 16-bit pair sweep (first tier when the y-drop keeps scores within 16
    bits), the same without its traced variant, and the 32-bit sweep give the
    same records, CIGARs and live cells; all equal the oracle.  Without the
    traced variant the executor replays the same cells as after the 32-bit
    sweep."""
    w = G.workload(2)
    idx = np.arange(2000)
    a, acig, sa = G.gpu_run(w, w.seeds[idx])
    monkeypatch.setenv("FZ_NO_PAIR", "1")
    b, bcig, sb = G.gpu_run(w, w.seeds[idx])
    monkeypatch.delenv("FZ_NO_PAIR")
    monkeypatch.setenv("FZ_TRACED", "0")
    c, ccig, sc = G.gpu_run(w, w.seeds[idx])
    monkeypatch.delenv("FZ_TRACED")
    assert np.array_equal(a, b) and np.array_equal(acig, bcig)
    assert np.array_equal(a, c) and np.array_equal(acig, ccig)
    assert sa.live_cells == sb.live_cells == sc.live_cells and sc.exec_cells == sb.exec_cells
    assert sb.traced == 0 and sc.traced == 0
    ores, ocig, ooff = G.oracle_run(w, w.seeds[idx])
    G.compare(w, w.seeds[idx], a, acig, ores, ocig, ooff, label="pair sweep")
    assert sa.live_cells == int(ores["live_cells"].sum())


def test_traced_sweep_on_long_alignments(monkeypatch):
    """The traced pair sweep (direction flags stored during the inspector, the
    warp walks its own best cell back) on chromosome-batch anchors, most of
    them predicted long: records and CIGARs equal the oracle's and those of
    the inspector + executor path (FZ_TRACED=0)."""
    w = G.workload(3)
    idx = G.sample_seeds(w, 3000, seed=31)
    monkeypatch.setenv("FZ_TRACE_MIN", "0")        # (a sample this small would not fill the traced warps)
    a, acig, sa, ores = _check(w, w.seeds[idx], label="traced sweep, chromosome anchors")
    assert sa.traced > 0.4 * sa.extensions
    assert sa.live_cells == int(ores["live_cells"].sum())
    monkeypatch.setenv("FZ_TRACED", "0")
    b, bcig, sb = G.gpu_run(w, w.seeds[idx])
    assert sb.traced == 0 and np.array_equal(a, b) and np.array_equal(acig, bcig)
    assert sa.eager + sum(sa.bin) + sa.traced == sa.extensions == sb.eager + sum(sb.bin)


def test_traced_overflow_uses_ring_checkpoints(monkeypatch):
    """Traced extensions whose band overflows the 384-row window continue in
    the 512-row tier and go to the executor, which splits their replay at the
    traced sweep's ring checkpoints (published on the overflow): records and
    CIGARs equal the oracle's, with small and default checkpoint intervals."""
    rng = np.random.default_rng(71)
    w, _ = _batch_from_pairs(_gap_run_pairs(rng, 40))
    monkeypatch.setenv("FZ_TRACE_ALL", "1")
    for every in ("32", None):
        if every:
            monkeypatch.setenv("FZ_CKPT_EVERY", every)
        else:
            monkeypatch.delenv("FZ_CKPT_EVERY", raising=False)
        gres, gcig, st, ores = _check(w, label=f"traced overflow, checkpoint interval {every}")
        assert st.retried > 0 and st.traced > 0
        assert st.live_cells == int(ores["live_cells"].sum())


@pytest.mark.parametrize("label,env", [("every extension traced", {"FZ_TRACE_ALL": "1"}),
                                       ("traced-run arena of 1,000 runs", {"FZ_TRACE_ALL": "1", "FZ_TRUNS_CAP": "1000"})])
def test_traced_sweep_everywhere(label, env, monkeypatch):
    """Every extension through the traced sweep: the edge cases (empty and
    one-base windows, ends at the corner and the bin edges, long gaps, every
    y-drop from 0 to none), the gap-run batch (band climbing and widening,
    512-row overflows) and random scorings; with a tiny traced-run arena most
    walked extensions do not fit and fall back to the executor, which then
    replays them from the origin."""
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    rng = np.random.default_rng(61)
    w, _ = _batch_from_pairs(_gap_run_pairs(rng, 30))
    gres, gcig, st, ores = _check(w, label=f"{label}: gap runs")
    assert st.traced + st.eager + sum(st.bin) == st.extensions
    if "FZ_TRUNS_CAP" not in env:
        assert st.traced > 0
    x = rng.integers(0, 4, 300).astype(np.uint8)
    pairs = [(np.zeros(0, np.uint8), np.zeros(0, np.uint8)), (x[:1], x[:1]), (x[:16], x[:16]), (x[:17], x[:16]),
             (x, x), (np.concatenate([x[:80], np.zeros(60, np.uint8), x[80:]]), x),
             (x[:100], np.concatenate([x[:50], x[60:100]])), (np.zeros(30, np.uint8), np.ones(30, np.uint8))]
    for L in (511, 512, 513):
        y = rng.integers(0, 4, L).astype(np.uint8)
        pairs.append((np.concatenate([y, np.zeros(40, np.uint8)]), np.concatenate([y, np.ones(40, np.uint8)])))
    w, _ = _batch_from_pairs(pairs)
    for yd in (0, 1, 429, 430, 5000, 9400):
        w2 = W.Workload(w.name, w.target, w.query, w.seeds, w.sub, w.gap_open, w.gap_extend, yd, w.max_len, w.mode)
        _check(w2, label=f"{label}: edge cases ydrop={yd}")
    for it in range(3):
        sub = rng.integers(-120, 121, size=(4, 4)).astype(np.int32)
        sub[np.arange(4), np.arange(4)] = rng.integers(20, 128, 4)
        pairs = []
        for _ in range(80):
            m = int(rng.integers(0, 400))
            t = rng.integers(0, 4, m).astype(np.uint8)
            q = W.mutate(rng, t[:int(rng.integers(0, m + 1))], rng.uniform(0, 0.3), rng.uniform(0, 0.05), 2.0)
            pairs.append((t, q))
        w, _ = _batch_from_pairs(pairs, sub=sub, o=int(rng.integers(0, 600)), e=int(rng.integers(1, 60)),
                                 ydrop=int(rng.choice([300, 2000, 9400])))
        _check(w, label=f"{label}: random scoring {it}")


def _gap_run_pairs(rng, n_pairs):
    """High-identity pairs with long gap runs: a deletion from the query moves
    the live band up one row per anti-diagonal (the window's base must follow
    every step), an insertion holds the band's bottom row while its top rises
    (the window keeps its base and may have to grow)."""
    pairs = []
    for k in range(n_pairs):
        t = rng.integers(0, 4, int(rng.integers(1200, 2400))).astype(np.uint8)
        q = W.mutate(rng, t, 0.03, 0.0, 1.0)
        cuts = np.sort(rng.choice(np.arange(150, min(t.size, q.size) - 150), size=3, replace=False))
        parts, last = [], 0
        for c in cuts:
            parts.append(q[last:c])
            glen = int(rng.integers(40, 260))
            if rng.random() < 0.5:
                parts.append(rng.integers(0, 4, glen).astype(np.uint8))     # insertion
                last = c
            else:
                last = min(q.size, c + glen)                                 # deletion
        parts.append(q[last:])
        q = np.concatenate(parts).astype(np.uint8)
        pairs.append((t, q) if k % 2 == 0 else (q, t))                       # gaps on either sequence
    return pairs


def test_gap_runs_move_the_band(monkeypatch):
    """Long gap runs (up to 260 bases, costing up to o + 260 e = 8,200 < ydrop)
    make the live band climb a row per step or hold its bottom while it widens:
    the pair sweep's keep/shift pairs leave early, take single steps with the
    top lane live, grow the window and overflow to the 512-row tier; with a
    checkpoint every 32 anti-diagonals the executor resumes segments at bases
    that trail the shift-by-one base.  Records and CIGARs equal the oracle's,
    and the 16-bit and 32-bit sweeps agree on every count."""
    rng = np.random.default_rng(47)
    w, _ = _batch_from_pairs(_gap_run_pairs(rng, 60))
    monkeypatch.setenv("FZ_CKPT_EVERY", "32")
    a, acig, st, ores = _check(w, label="gap runs")
    assert st.live_cells == int(ores["live_cells"].sum())
    monkeypatch.setenv("FZ_NO_PAIR", "1")
    b, bcig, sb = G.gpu_run(w)
    monkeypatch.delenv("FZ_NO_PAIR")
    monkeypatch.setenv("FZ_TRACED", "0")
    c, ccig, sc = G.gpu_run(w)
    assert np.array_equal(a, b) and np.array_equal(acig, bcig)
    assert np.array_equal(a, c) and np.array_equal(acig, ccig)
    assert st.live_cells == sb.live_cells == sc.live_cells and sc.exec_cells == sb.exec_cells
    assert st.retried == sb.retried == sc.retried


@pytest.mark.parametrize("ydrop", [20000, 20252])
def test_pair_sweep_at_its_range_limit(ydrop, monkeypatch):
    """The 16-bit pair sweep at the largest y-drops it takes with HOXD70 and
    o = 1500, e = 300 (ydrop + 2048 + 4 (o + e + max|M|) <= 30000; steep gaps keep
    the band inside the 384-row window): little or no slack, so the stored
    values move at nearly every rise of the best score, and live values reach
    the top of the 16-bit range.  Long high-identity pairs drive scores far
    from 0; both sweeps and the oracle must agree."""
    rng = np.random.default_rng(41)
    pairs = []
    for _ in range(40):
        t = rng.integers(0, 4, int(rng.integers(500, 3000))).astype(np.uint8)
        q = W.mutate(rng, t, rng.uniform(0.0, 0.15), rng.uniform(0.0, 0.02), 3.0)
        pairs.append((t, q))
    w, _ = _batch_from_pairs(pairs, o=1500, e=300, ydrop=ydrop)
    a, acig, st, ores = _check(w, label=f"pair range limit ydrop={ydrop}")
    monkeypatch.setenv("FZ_NO_PAIR", "1")
    b, bcig, sb = G.gpu_run(w)
    assert np.array_equal(a, b) and np.array_equal(acig, bcig) and st.live_cells == sb.live_cells


def test_two_sided_combination():
    """fz_combine on two-sided anchors of the chromosome workload against the
    oracle's combination of its one-sided results."""
    import oracle
    from gapped_smith_waterman_gb300 import fz
    w = G.workload(3)
    idx = G.sample_seeds(w, 300, seed=21)
    seeds = w.seeds[idx]
    ext = fz.Extender.for_workload(w)
    try:
        aln, cig = ext.extend_and_combine(w, seeds)
    finally:
        ext.close()
    ores, ocig, ooff = G.oracle_run(w, seeds)
    exp = oracle.combine(seeds, ores, ocig, ooff)
    assert len(aln) == len(exp)
    for k, (score, ts, qs, te, qe, runs) in enumerate(exp):
        a = aln[k]
        assert (int(a["score"]), int(a["t_start"]), int(a["q_start"]), int(a["t_end"]), int(a["q_end"])) == \
            (score, ts, qs, te, qe), k
        got = cig[int(a["cigar_off"]):int(a["cigar_off"]) + int(a["cigar_len"])]
        assert np.array_equal(got, runs), k
    # packed in seed order
    assert np.array_equal(aln["cigar_off"][1:], (aln["cigar_off"] + aln["cigar_len"])[:-1])


def test_chunked_executor(monkeypatch):
    w = G.workload(1)
    monkeypatch.setenv("FZ_TRACED", "0")            # (256 bp windows would all take the traced sweep)
    a, acig, sa = G.gpu_run(w)
    monkeypatch.setenv("FZ_TRACE_CAP", str(1 << 20))
    b, bcig, sb = G.gpu_run(w)
    assert np.array_equal(a, b) and np.array_equal(acig, bcig)


def test_context_reuse_and_growth():
    from gapped_smith_waterman_gb300 import fz
    w = G.workload(1)
    ext = fz.Extender.for_workload(w)
    try:
        r1 = ext.extend_workload(w, w.seeds[:10])
        r2 = ext.extend_workload(w, w.seeds)
        r3 = ext.extend_workload(w, w.seeds[:10])
        assert np.array_equal(r1[0], r3[0])
        assert np.array_equal(r1[0], r2[0][:20])
        r0 = ext.extend_workload(w, w.seeds[:0])
        assert r0[0].size == 0
    finally:
        ext.close()


def test_error_codes(monkeypatch):
    from gapped_smith_waterman_gb300 import fz
    with pytest.raises(fz.FzError) as ei:
        fz.fz_create(W.HOXD70, 400, 0, 9400, 100)
    assert ei.value.status == fz.FZ_ERR_ARG
    with pytest.raises(fz.FzError):
        fz.fz_create(W.HOXD70, 400, 30, -5, 100)
    with pytest.raises(fz.FzError):
        fz.fz_create(W.HOXD70 * 2, 400, 30, 9400, 100, fz.FZ_LOCAL)
    w = G.workload(1)
    ext = fz.Extender.for_workload(w)
    try:
        monkeypatch.setenv("FZ_FAULT", "alloc")
        with pytest.raises(fz.FzError) as ei:
            ext.extend_workload(w, w.seeds[:5])
        assert ei.value.status == fz.FZ_ERR_OOM
        monkeypatch.delenv("FZ_FAULT")
        r = ext.extend_workload(w, w.seeds[:5])
        assert r[0].size == 10
    finally:
        ext.close()
