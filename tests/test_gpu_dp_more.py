"""GPU parity of the batched edit distance and dynamic time warping (the DPX
article's other dynamic programs, section 1.3) against the CPU oracle: every
pair, exact integer results, including the article's batch sizes (section
4.1), lengths at the 1,024-column strip edges, empty pairs and the limits."""
import numpy as np
import pytest

from gapped_smith_waterman_gb300 import workloads as W

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


def _run(kind, a, b, pairs):
    from gapped_smith_waterman_gb300 import fz
    return fz.dp_pairs_device(kind, a, b, pairs)


def _oracle(kind, a, b, pairs):
    import oracle
    return oracle.pairs_batch(oracle.edit_distance if kind == "edit" else oracle.dtw, a, b, pairs)


def _mixed_pairs(kind, rng, lens):
    a_parts, b_parts, la, lb = [], [], [], []
    for m, n in lens:
        if kind == "edit":
            a = rng.integers(0, 4, m).astype(np.uint8)
            b = W.mutate(rng, a, 0.15, 0.02, 2.0)[:n] if rng.random() < 0.5 else rng.integers(0, 4, n).astype(np.uint8)
            b = np.concatenate([b, rng.integers(0, 4, n - b.size).astype(np.uint8)]) if b.size < n else b
        else:
            a = W.random_walk(rng, m, int(rng.integers(1, 200)))
            b = W.random_walk(rng, n, int(rng.integers(1, 200)))
        a_parts.append(a)
        b_parts.append(b[:n])
        la.append(m)
        lb.append(n)
    dt = np.uint8 if kind == "edit" else np.int32
    a = np.concatenate(a_parts).astype(dt) if a_parts else np.zeros(0, dt)
    b = np.concatenate(b_parts).astype(dt) if b_parts else np.zeros(0, dt)
    return a, b, W.dp_pairs(la, lb)


EDGE_LENS = [(0, 0), (0, 5), (7, 0), (1, 1), (1, 1500), (1500, 1), (31, 33), (32, 32), (1023, 1024),
             (1024, 1023), (1025, 1025), (2047, 2049), (3000, 2100), (4096, 4096), (4096, 1), (1, 4096)]


@pytest.mark.parametrize("kind", ["edit", "dtw"])
def test_every_pair_against_the_oracle(kind):
    rng = np.random.default_rng(11 if kind == "edit" else 12)
    lens = EDGE_LENS + [(int(rng.integers(0, 3000)), int(rng.integers(0, 3000))) for _ in range(60)]
    a, b, pairs = _mixed_pairs(kind, rng, lens)
    got = _run(kind, a, b, pairs)
    want = _oracle(kind, a, b, pairs)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{kind}: {bad.size} pairs differ, first {bad[0]}: lens {lens[bad[0]]} gpu {got[bad[0]]} oracle {want[bad[0]]}"


@pytest.mark.parametrize("kind", ["edit", "dtw"])
def test_the_articles_batch_sizes(kind):
    w = W.make_edit_batch() if kind == "edit" else W.make_dtw_batch()
    got = _run(kind, w.a, w.b, w.pairs)
    want = _oracle(kind, w.a, w.b, w.pairs)
    assert np.array_equal(got, want)
    if kind == "edit":
        # related pairs are far closer than unrelated ones
        assert got[0::2].mean() < 0.5 * got[1::2].mean()


def test_limits_and_bad_samples():
    rng = np.random.default_rng(13)
    a = rng.integers(0, 4, 9000).astype(np.uint8)
    b = rng.integers(0, 4, 9000).astype(np.uint8)
    pairs = W.dp_pairs([4097, 10, 10], [10, 4097, 10])
    pairs["a_pos"][2] = 8995                      # runs past the end of a
    assert list(_run("edit", a, b, pairs)) == [-2, -2, -2]
    x = np.zeros(100, np.int32)
    y = np.zeros(100, np.int32)
    x[50] = 40000                                 # a sample outside [-32767, 32767]
    p2 = W.dp_pairs([60, 40], [60, 40])
    p2["a_pos"][1] = 60
    got = _run("dtw", x, y, p2)
    assert got[0] == -2 and got[1] == 0


def test_argument_errors():
    from gapped_smith_waterman_gb300 import fz
    with pytest.raises(fz.FzError) as ei:
        fz.fz_edit_distance_batch(0, 0, 0, 0, 0, 3, 0)
    assert ei.value.status == fz.FZ_ERR_ARG
    with pytest.raises(fz.FzError) as ei:
        fz.fz_dtw_batch(0, 10, 0, 0, 0, 1, 0)
    assert ei.value.status == fz.FZ_ERR_ARG
    fz.fz_edit_distance_batch(0, 0, 0, 0, 0, 0, 0)     # no pairs: nothing to do
